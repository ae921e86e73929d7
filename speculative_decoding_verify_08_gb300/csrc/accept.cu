// accept.cu -- exact Leviathan-Chen acceptance of K drafts per round.
//
// Rule ("The fastest way to run local LLMs on a Mac", section "Why exact
// acceptance matters"): accept draft x with probability min(1, p(x)/q(x)),
// i.e. iff u * q(x) < p(x); on the first rejection resample from (p - q)+ and
// stop; if every draft is accepted sample a bonus token from the last target
// row.  p and q are truncated identically ("Speculative decoding and MTP on
// Apple silicon", Facts): temperature, then top-k (ties with the k-th logit
// kept), then top-p (a token is kept while the mass of strictly more likely
// tokens is below top_p).
//
// Two kernels:
//  1. select: one CTA per logits row streams the row once from HBM and keeps
//     a shared-memory buffer of candidates above a running threshold; when
//     the buffer fills it radix-selects the k-th largest key and drops the
//     rest.  The exact top-k set (with ties) is written out in index order.
//     Keys are the order-preserving integer image of the fp32 logit, so the
//     set equals the one selected on l = z/T in fp64.
//  2. chain: one CTA per round evaluates the truncated distributions over the
//     candidates in fp64 (exp, sums and divisions in the same order as the
//     CPU definition: index order for normalising sums, decreasing logit for
//     the nucleus mass) and runs the sequential accept / residual / bonus
//     chain.
// With top_k off and V <= 2048 the whole row is the candidate list and the
// select pass is skipped.
#include "common.cuh"

namespace sv {
namespace acc {

constexpr int SEL_THREADS = 512;
constexpr int SEL_PER_THREAD = 8;
constexpr int SEL_CHUNK = SEL_THREADS * SEL_PER_THREAD;  // 4096
constexpr int SEL_BUF = 2 * SEL_CHUNK;                   // 8192
constexpr int CAND_MAX = 2048;
constexpr int MAX_TOPK = 1024;
constexpr int ROW_BYTES = 16 + 8 * CAND_MAX;  // count + values + indices
constexpr int CHAIN_THREADS = 128;
constexpr int MAX_K = 32;

__device__ __forceinline__ uint32_t fkey(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0 and +0 compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float keyf(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

template <typename T>
__device__ __forceinline__ float load_logit(const T *p, long long i);
template <>
__device__ __forceinline__ float load_logit<float>(const float *p, long long i) {
  return __ldcs(p + i);
}
template <>
__device__ __forceinline__ float load_logit<__nv_bfloat16>(const __nv_bfloat16 *p, long long i) {
  const unsigned short b = __ldcs(reinterpret_cast<const unsigned short *>(p) + i);
  return __uint_as_float((uint32_t)b << 16);
}

struct SelShared {
  uint32_t key[SEL_BUF];
  uint32_t idx[SEL_BUF];
  int hist[256];
  int cnt, cnt2, sel, krem;
  uint32_t tau;
};

// Row (round r, j): j <= K target row j, else draft row j-K-1.
template <typename T>
__device__ __forceinline__ const T *row_ptr(const T *tgt, const T *drf, int r, int j, int K, int V) {
  return j <= K ? tgt + ((size_t)r * (K + 1) + j) * V : drf + ((size_t)r * K + (j - K - 1)) * V;
}

// Keep the entries whose key is >= the k-th largest key of the buffer.
__device__ void compact(SelShared &s, int k) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int n = s.cnt;
  if (n <= k) return;
  uint32_t prefix = 0, pmask = 0;
  int krem = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += SEL_THREADS) s.hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += SEL_THREADS) {
      const uint32_t key = s.key[i];
      if ((key & pmask) == prefix) atomicAdd(&s.hist[(key >> shift) & 255], 1);
    }
    __syncthreads();
    if (tid < 32) {
      // lane l holds digits 255-8l .. 248-8l (descending)
      int c[8], tot = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        c[e] = s.hist[255 - 8 * lane - e];
        tot += c[e];
      }
      int incl = tot;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      const int excl = incl - tot;
      const unsigned hit = __ballot_sync(0xffffffffu, incl >= krem);
      const int first = __ffs(hit) - 1;
      if (lane == first) {
        int cum = excl;
        for (int e = 0; e < 8; ++e) {
          if (cum + c[e] >= krem) {
            s.sel = 255 - 8 * lane - e;
            s.krem = krem - cum;
            break;
          }
          cum += c[e];
        }
      }
    }
    __syncthreads();
    prefix |= (uint32_t)s.sel << shift;
    pmask |= 0xFFu << shift;
    krem = s.krem;
    __syncthreads();
  }
  const uint32_t kth = prefix;
  // in-place compaction through registers
  uint32_t kk[SEL_BUF / SEL_THREADS], ii[SEL_BUF / SEL_THREADS];
#pragma unroll
  for (int e = 0; e < SEL_BUF / SEL_THREADS; ++e) {
    const int i = tid + e * SEL_THREADS;
    kk[e] = i < n ? s.key[i] : 0u;
    ii[e] = i < n ? s.idx[i] : 0u;
  }
  if (tid == 0) s.cnt2 = 0;
  __syncthreads();
#pragma unroll
  for (int e = 0; e < SEL_BUF / SEL_THREADS; ++e) {
    const int i = tid + e * SEL_THREADS;
    const bool keep = i < n && kk[e] >= kth;
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    if (m) {
      const int leader = __ffs(m) - 1;
      int base = 0;
      if (lane == leader) base = atomicAdd(&s.cnt2, __popc(m));
      base = __shfl_sync(0xffffffffu, base, leader);
      if (keep) {
        const int pos = base + __popc(m & ((1u << lane) - 1u));
        s.key[pos] = kk[e];
        s.idx[pos] = ii[e];
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    s.cnt = s.cnt2;
    s.tau = kth;
  }
  __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(SEL_THREADS)
    select_kernel(const T *__restrict__ tgt, const T *__restrict__ drf, int K, int V, int k,
                  uint8_t *__restrict__ ws, unsigned *err) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelShared &s = *reinterpret_cast<SelShared *>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31;
  const int row = blockIdx.x;
  const int r = row / (2 * K + 1), j = row % (2 * K + 1);
  pdl_launch_dependents();
  pdl_wait();
  const T *z = row_ptr(tgt, drf, r, j, K, V);
  if (tid == 0) {
    s.cnt = 0;
    s.tau = 0u;
  }
  __syncthreads();
  for (long long cb = 0; cb < V; cb += SEL_CHUNK) {
    const uint32_t tau = s.tau;
    float v[SEL_PER_THREAD];
#pragma unroll
    for (int e = 0; e < SEL_PER_THREAD; ++e) {
      const long long i = cb + (long long)e * SEL_THREADS + tid;
      v[e] = i < V ? load_logit(z, i) : 0.f;
    }
#pragma unroll
    for (int e = 0; e < SEL_PER_THREAD; ++e) {
      const long long i = cb + (long long)e * SEL_THREADS + tid;
      const uint32_t key = fkey(v[e]);
      const bool pass = i < V && key >= tau;
      const unsigned m = __ballot_sync(0xffffffffu, pass);
      if (m) {
        const int leader = __ffs(m) - 1;
        int base = 0;
        if (lane == leader) base = atomicAdd(&s.cnt, __popc(m));
        base = __shfl_sync(0xffffffffu, base, leader);
        if (pass) {
          const int pos = base + __popc(m & ((1u << lane) - 1u));
          s.key[pos] = key;
          s.idx[pos] = (uint32_t)i;
        }
      }
    }
    __syncthreads();
    if (s.cnt > SEL_BUF - SEL_CHUNK) {
      compact(s, k);
      if (s.cnt > SEL_BUF - SEL_CHUNK) {  // ties fill the buffer
        if (tid == 0) atomicOr(err, ERR_OVERFLOW);
        break;
      }
    }
  }
  compact(s, k);
  const int n = s.cnt;
  uint8_t *out = ws + (size_t)row * ROW_BYTES;
  if (n > CAND_MAX || n > SEL_BUF - SEL_CHUNK) {
    if (tid == 0) {
      atomicOr(err, ERR_OVERFLOW);
      *reinterpret_cast<int *>(out) = -1;
    }
    return;
  }
  // bitonic sort by index (ascending); pad with 0xFFFFFFFF
  int P2 = 1;
  while (P2 < n) P2 <<= 1;
  for (int i = n + tid; i < P2; i += SEL_THREADS) {
    s.idx[i] = 0xFFFFFFFFu;
    s.key[i] = 0u;
  }
  __syncthreads();
  for (int size = 2; size <= P2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < P2; i += SEL_THREADS) {
        const int p = i ^ stride;
        if (p > i) {
          const bool asc = (i & size) == 0;
          const uint32_t a = s.idx[i], b = s.idx[p];
          if ((a > b) == asc) {
            s.idx[i] = b;
            s.idx[p] = a;
            const uint32_t t = s.key[i];
            s.key[i] = s.key[p];
            s.key[p] = t;
          }
        }
      }
      __syncthreads();
    }
  }
  float *vals = reinterpret_cast<float *>(out + 16);
  int *idxs = reinterpret_cast<int *>(out + 16 + 4 * CAND_MAX);
  for (int i = tid; i < n; i += SEL_THREADS) {
    vals[i] = keyf(s.key[i]);
    idxs[i] = (int)s.idx[i];
  }
  if (tid == 0) *reinterpret_cast<int *>(out) = n;
}

// ------------------------------------------------------------- chain ---
struct ChainParams {
  const void *tgt, *drf;
  int bf16;
  const int32_t *drafts;
  const float *u;
  int32_t *out_tok, *out_n;
  const uint8_t *ws;  // select output (null when the whole row is the list)
  int R, K, V;
  double T, top_p;
  unsigned *err;
};

struct List {
  int *idx;
  float *val;
  double *p;
  int n;
};

struct ChainShared {
  int accept;
};

__device__ __forceinline__ float logit_at(const ChainParams &cp, int r, int j, int i) {
  const bool is_t = j <= cp.K;
  const size_t off = is_t ? ((size_t)r * (cp.K + 1) + j) * cp.V
                          : ((size_t)r * cp.K + (j - cp.K - 1)) * cp.V;
  const void *base = is_t ? cp.tgt : cp.drf;
  if (cp.bf16) {
    const unsigned short b = static_cast<const unsigned short *>(base)[off + i];
    return __uint_as_float((uint32_t)b << 16);
  }
  return static_cast<const float *>(base)[off + i];
}

// Load row (r, j)'s candidate list into L (index order); returns count, or
// -1 if the select pass overflowed.
__device__ int load_list(const ChainParams &cp, int r, int j, List &L) {
  const int tid = threadIdx.x;
  if (cp.ws) {
    const uint8_t *in = cp.ws + ((size_t)r * (2 * cp.K + 1) + j) * ROW_BYTES;
    const int n = *reinterpret_cast<const int *>(in);
    if (n < 0) return -1;
    const float *vals = reinterpret_cast<const float *>(in + 16);
    const int *idxs = reinterpret_cast<const int *>(in + 16 + 4 * CAND_MAX);
    for (int i = tid; i < n; i += CHAIN_THREADS) {
      L.val[i] = vals[i];
      L.idx[i] = idxs[i];
    }
    return n;
  }
  for (int i = tid; i < cp.V; i += CHAIN_THREADS) {
    L.val[i] = logit_at(cp, r, j, i);
    L.idx[i] = i;
  }
  return cp.V;
}

// Block-wide max of doubles.
__device__ double block_max(double v, double *scratch) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  for (int off = 16; off > 0; off >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, off));
  __syncthreads();
  if (lane == 0) scratch[w] = v;
  __syncthreads();
  double m = scratch[0];
  for (int i = 1; i < CHAIN_THREADS / 32; ++i) m = fmax(m, scratch[i]);
  __syncthreads();
  return m;
}

// Truncated distribution over the list (written to L.p, index order).
__device__ void dist(const ChainParams &cp, List &L, int *perm, unsigned char *keep,
                     double *scratch, double *shared_sum) {
  const int tid = threadIdx.x;
  const int n = L.n;
  if (cp.T == 0.0) {
    // the list is the set of logits tied at the maximum, in index order
    for (int i = tid; i < n; i += CHAIN_THREADS) L.p[i] = (i == 0) ? 1.0 : 0.0;
    __syncthreads();
    return;
  }
  double lm = -INFINITY;
  for (int i = tid; i < n; i += CHAIN_THREADS) lm = fmax(lm, (double)L.val[i] / cp.T);
  lm = block_max(lm, scratch);
  for (int i = tid; i < n; i += CHAIN_THREADS) L.p[i] = exp((double)L.val[i] / cp.T - lm);
  __syncthreads();
  if (tid == 0) {
    double Z = 0.0;
    for (int i = 0; i < n; ++i) Z += L.p[i];
    *shared_sum = Z;
  }
  __syncthreads();
  const double Z = *shared_sum;
  for (int i = tid; i < n; i += CHAIN_THREADS) L.p[i] = L.p[i] / Z;
  __syncthreads();
  if (!(cp.top_p < 1.0)) return;

  // order by (logit desc, index asc): bitonic sort of a permutation
  int P2 = 1;
  while (P2 < n) P2 <<= 1;
  for (int i = tid; i < P2; i += CHAIN_THREADS) perm[i] = i < n ? i : -1;
  __syncthreads();
  for (int size = 2; size <= P2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < P2; i += CHAIN_THREADS) {
        const int p = i ^ stride;
        if (p > i) {
          const bool asc = (i & size) == 0;
          const int a = perm[i], b = perm[p];
          // "a before b": a valid and (b invalid or val larger or equal val, smaller idx)
          bool a_first;
          if (a < 0) a_first = false;
          else if (b < 0) a_first = true;
          else a_first = (L.val[a] > L.val[b]) || (L.val[a] == L.val[b] && L.idx[a] < L.idx[b]);
          if (a_first != asc) {
            perm[i] = b;
            perm[p] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  if (tid == 0) {
    double above = 0.0;
    int a = 0;
    while (a < n) {
      int b = a;
      while (b < n && L.val[perm[b]] == L.val[perm[a]]) ++b;
      const unsigned char kp = above < cp.top_p ? 1 : 0;
      for (int c = a; c < b; ++c) keep[perm[c]] = kp;
      for (int c = a; c < b; ++c) above += L.p[perm[c]];
      a = b;
    }
    double S = 0.0;
    for (int i = 0; i < n; ++i)
      if (keep[i]) S += L.p[i];
    *shared_sum = S;
  }
  __syncthreads();
  const double S = *shared_sum;
  for (int i = tid; i < n; i += CHAIN_THREADS) L.p[i] = keep[i] ? L.p[i] / S : 0.0;
  __syncthreads();
}

__device__ double lookup(const List &L, int x) {
  int lo = 0, hi = L.n - 1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    const int v = L.idx[mid];
    if (v == x) return L.p[mid];
    if (v < x) lo = mid + 1;
    else hi = mid - 1;
  }
  return 0.0;
}

// First index whose running sum of w (index order) exceeds t; if none, the
// last index with w > 0 (0 if there is none).
__device__ int icdf(const List &L, const double *w, double t) {
  double c = 0.0;
  int last_pos = 0;
  for (int i = 0; i < L.n; ++i) {
    c += w[i];
    if (w[i] > 0.0) last_pos = L.idx[i];
    if (c > t) return L.idx[i];
  }
  return last_pos;
}

__global__ void __launch_bounds__(CHAIN_THREADS) chain_kernel(const ChainParams cp) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int cap = cp.ws ? CAND_MAX : cp.V;
  double *pP = reinterpret_cast<double *>(smem_raw);
  double *pQ = pP + cap;
  double *wv = pQ + cap;
  double *scratch = wv + cap;  // 8 doubles
  double *shared_sum = scratch + 8;
  float *vP = reinterpret_cast<float *>(shared_sum + 2);
  float *vQ = vP + cap;
  int *iP = reinterpret_cast<int *>(vQ + cap);
  int *iQ = iP + cap;
  int *perm = iQ + cap;  // 2*cap (power-of-two padding)
  unsigned char *keep = reinterpret_cast<unsigned char *>(perm + 2 * cap);
  __shared__ ChainShared cs;

  const int r = blockIdx.x, tid = threadIdx.x;
  const int K = cp.K;
  pdl_launch_dependents();
  pdl_wait();
  List P{iP, vP, pP, 0}, Q{iQ, vQ, pQ, 0};
  int32_t *tok = cp.out_tok + (size_t)r * (K + 1);
  const float *u = cp.u + (size_t)r * (K + 1);
  for (int i = tid; i <= K; i += CHAIN_THREADS) tok[i] = -1;
  __syncthreads();

  int n_acc = K;
  bool bad = false;  // a candidate list overflowed in the select pass (uniform)
  for (int i = 0; i < K; ++i) {
    const int np = load_list(cp, r, i, P);
    const int nq = load_list(cp, r, K + 1 + i, Q);
    if (np < 0 || nq < 0) {
      bad = true;
      break;
    }
    P.n = np;
    Q.n = nq;
    __syncthreads();
    dist(cp, P, perm, keep, scratch, shared_sum);
    dist(cp, Q, perm, keep, scratch, shared_sum);
    if (tid == 0) {
      const int x = cp.drafts[(size_t)r * K + i];
      const double px = lookup(P, x), qx = lookup(Q, x);
      cs.accept = ((double)u[i] * qx < px) ? 1 : 0;
      if (cs.accept) {
        tok[i] = x;
      } else {
        // residual (p - q)+ over p's candidates, index order (q by merge)
        double W = 0.0;
        int jq = 0;
        for (int jp = 0; jp < P.n; ++jp) {
          const int id = P.idx[jp];
          while (jq < Q.n && Q.idx[jq] < id) ++jq;
          const double qj = (jq < Q.n && Q.idx[jq] == id) ? Q.p[jq] : 0.0;
          const double d = P.p[jp] - qj;
          wv[jp] = d > 0.0 ? d : 0.0;
          W += wv[jp];
        }
        if (W == 0.0) {
          for (int jp = 0; jp < P.n; ++jp) wv[jp] = P.p[jp];
          W = 1.0;
        }
        tok[i] = icdf(P, wv, (double)u[K] * W);
      }
    }
    __syncthreads();
    if (!cs.accept) {
      n_acc = i;
      break;
    }
  }
  if (!bad && n_acc == K) {
    const int np = load_list(cp, r, K, P);
    if (np < 0) {
      bad = true;
    } else {
      P.n = np;
      __syncthreads();
      dist(cp, P, perm, keep, scratch, shared_sum);
      if (tid == 0) tok[K] = icdf(P, P.p, (double)u[K]);
    }
  }
  __syncthreads();
  if (tid == 0) {
    if (bad) {
      cp.out_n[r] = -1;
      atomicOr(cp.err, ERR_OVERFLOW);
    } else {
      cp.out_n[r] = n_acc;
    }
  }
}

static size_t chain_smem(int cap) {
  return (size_t)cap * (8 * 3 + 4 * 2 + 4 * 2 + 4 * 2 + 1) + 8 * 10 + 16;
}

}  // namespace acc
}  // namespace sv

using namespace sv;

extern "C" {

size_t spec_accept_workspace_bytes(int R, int K, int V) {
  if (R < 1 || K < 1 || V < 1) return 0;
  return (size_t)R * (2 * K + 1) * acc::ROW_BYTES;
}

sv_status spec_accept(const void *target_logits, const void *draft_logits, sv_dtype logit_dtype,
                      const int32_t *draft_tokens, const float *uniforms, sv_sampling_params params,
                      int R, int K, int V, int32_t *out_tokens, int32_t *out_num_accepted,
                      void *workspace, size_t ws_bytes, sv_stream_t stream) {
  if (!target_logits || !draft_logits || !draft_tokens || !uniforms || !out_tokens || !out_num_accepted)
    return SV_ERR_INVALID_ARG;
  if (R < 1 || K < 1 || V < 1) return SV_ERR_INVALID_ARG;
  if (logit_dtype != SV_F32 && logit_dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  const float T = params.temperature, tp = params.top_p;
  if (!(T >= 0.f) || !(T < INFINITY)) return SV_ERR_INVALID_ARG;
  if (!(tp > 0.f && tp <= 1.f)) return SV_ERR_INVALID_ARG;
  if (params.top_k < 0) return SV_ERR_INVALID_ARG;
  if (K > acc::MAX_K) return SV_ERR_UNSUPPORTED;
  int k = 0;
  bool whole_row = false;
  if (T == 0.f) {
    k = 1;
  } else if (params.top_k > 0 && params.top_k < V) {
    if (params.top_k > acc::MAX_TOPK) return SV_ERR_UNSUPPORTED;
    k = params.top_k;
  } else {
    if (V > acc::CAND_MAX) return SV_ERR_UNSUPPORTED;
    whole_row = true;
  }
  const size_t need = whole_row ? 0 : spec_accept_workspace_bytes(R, K, V);
  if (need > 0 && (!workspace || ws_bytes < need)) return SV_ERR_WORKSPACE;
  unsigned *err = device_error_word();
  if (!err) return SV_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int bf = logit_dtype == SV_BF16;
  cudaError_t e = cudaSuccess;
  if (!whole_row) {
    const long long rows = (long long)R * (2 * K + 1);
    if (rows > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
    const size_t sm = sizeof(acc::SelShared);
    if (bf)
      e = launch(acc::select_kernel<__nv_bfloat16>, dim3((unsigned)rows), dim3(acc::SEL_THREADS), sm, s,
                 static_cast<const __nv_bfloat16 *>(target_logits),
                 static_cast<const __nv_bfloat16 *>(draft_logits), K, V, k,
                 static_cast<uint8_t *>(workspace), err);
    else
      e = launch(acc::select_kernel<float>, dim3((unsigned)rows), dim3(acc::SEL_THREADS), sm, s,
                 static_cast<const float *>(target_logits), static_cast<const float *>(draft_logits), K,
                 V, k, static_cast<uint8_t *>(workspace), err);
    if (e != cudaSuccess) return SV_ERR_CUDA;
  }
  acc::ChainParams cp{};
  cp.tgt = target_logits;
  cp.drf = draft_logits;
  cp.bf16 = bf;
  cp.drafts = draft_tokens;
  cp.u = uniforms;
  cp.out_tok = out_tokens;
  cp.out_n = out_num_accepted;
  cp.ws = whole_row ? nullptr : static_cast<const uint8_t *>(workspace);
  cp.R = R;
  cp.K = K;
  cp.V = V;
  cp.T = (double)T;
  cp.top_p = (double)tp;
  cp.err = err;
  const int cap = whole_row ? V : acc::CAND_MAX;
  e = launch(acc::chain_kernel, dim3(R), dim3(acc::CHAIN_THREADS), acc::chain_smem(cap), s, cp);
  return from_cuda(e);
}

}  // extern "C"
