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
// Three kernels:
//  1. select: CTAs per logits row stream the row once from HBM and keep a
//     shared-memory buffer of candidates above a running threshold; when the
//     buffer fills they radix-select the k-th largest key and drop the rest.
//     Keys are the order-preserving integer image of the fp32 logit, so the
//     set equals the one selected on l = z/T in fp64.  The CTA that finishes
//     a row writes its exact top-k set (with ties) in index order.
//  2. dist: one warp per row evaluates the truncated distribution over the
//     row's candidates in fp64 (exp, sums and divisions in the same order as
//     the CPU definition: index order for normalising sums, decreasing logit
//     for the nucleus mass) -- every row of every round in parallel.
//  3. chain: one warp per round runs the sequential accept / residual /
//     bonus chain on those distributions.
// With the lm_head fused (qmm_small_m_topk writes every CTA's top-k of its
// own vocabulary columns), spec_accept_lists replaces the select pass of the
// target rows by a merge of those lists (merge_lists_kernel); the draft rows
// come from spec_accept_draft_select (the select pass over the draft rows
// only) or from the drafter's own lists.
// This path serves temperature 0 and top-k of at most 1024 below V; every
// other setting (top-k off, top-k >= V, larger top-k) takes the
// whole-vocabulary path of accept_whole.cu.
#include "accept_common.cuh"

namespace sv {
namespace acc {

constexpr int SEL_THREADS = 256;
constexpr int SEL_PER_THREAD = 8;
constexpr int SEL_CHUNK = SEL_THREADS * SEL_PER_THREAD;  // 2048 logits per step
// chunks between the CTA's barriers (2, with a 6144-entry buffer, measured 4%
// slower for the 256-round batch than a barrier after every chunk)
constexpr int SEL_GROUP = 1;
constexpr int SEL_BUF = (SEL_GROUP + 1) * SEL_CHUNK;     // 4096 buffered candidates
constexpr int SEL_PF = 4;  // chunk prefetched into L2 (ahead of the current one)
constexpr int CAND_MAX = 2048;
// a list row: count, then either (chunk lists) keys and indices, or (final
// lists) indices, fp64 probabilities, fp32 logits, and scratch for the
// distribution of a long list (sort permutation, keep flags)
constexpr int ROW_BYTES = 16 + 21 * CAND_MAX;
constexpr int FINAL_P_OFF = 16 + 4 * CAND_MAX;
constexpr int FINAL_V_OFF = 16 + 12 * CAND_MAX;
constexpr int FINAL_PERM_OFF = 16 + 16 * CAND_MAX;
constexpr int FINAL_KEEP_OFF = 16 + 20 * CAND_MAX;
constexpr int DIST_WARPS = 1;   // rows per dist CTA (one: spread the fp64 work over SMs)
constexpr int DIST_SCAP = 256;  // lists up to this long are evaluated in shared memory
constexpr int CHAIN_THREADS = 32;             // one warp per round

struct SelLayout {
  unsigned *counters;  // [rows], last-arriver merge
  uint8_t *final;      // [rows][ROW_BYTES]: count, indices, probabilities, logits (index order)
  uint8_t *chunks;     // [rows][C][ROW_BYTES]: count, keys, indices (any order)
};

static size_t sel_bytes(long long rows, int C) {
  const size_t counters = ((size_t)rows * 4 + 255) / 256 * 256;
  return counters + (size_t)rows * ROW_BYTES + (C > 1 ? (size_t)rows * C * ROW_BYTES : 0);
}


struct SelShared {
  uint32_t key[SEL_BUF];
  uint32_t idx[SEL_BUF];
  int hist[256];
  int cnt, cnt2, sel, krem;
  uint32_t tau;
};

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
  // in-place compaction, 2048 entries at a time in order: an entry moves only
  // to a lower position, so a batch read into registers before any of its
  // writes never overwrites an entry not yet read
  constexpr int E = 8;
  if (tid == 0) s.cnt2 = 0;
  __syncthreads();
  for (int b0 = 0; b0 < n; b0 += E * SEL_THREADS) {
    uint32_t kk[E], ii[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = b0 + tid + e * SEL_THREADS;
      kk[e] = i < n ? s.key[i] : 0u;
      ii[e] = i < n ? s.idx[i] : 0u;
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int i = b0 + tid + e * SEL_THREADS;
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
  }
  if (tid == 0) {
    s.cnt = s.cnt2;
    s.tau = kth;
  }
  __syncthreads();
}

struct List {
  int *idx;
  float *val;
  double *p;
  int n;
};

// Truncated distribution over the list, written to L.p (index order).  The
// floating-point operations follow the CPU definition one for one: l = z/T,
// e = exp(l - max), Z summed in index order, p = e/Z; top-p masses summed in
// decreasing-logit order (ties as one group), the kept total in index order.
__device__ void dist(double T, double top_p, List &L, int *perm, unsigned char *keep) {
  const int lane = threadIdx.x & 31;
  const int n = L.n;
  if (T == 0.0) {
    // the list is the set of logits tied at the maximum, in index order
    for (int i = lane; i < n; i += 32) L.p[i] = (i == 0) ? 1.0 : 0.0;
    __syncwarp();
    return;
  }
  double lm = -INFINITY;
  for (int i = lane; i < n; i += 32) lm = fmax(lm, (double)L.val[i] / T);
  for (int off = 16; off > 0; off >>= 1) lm = fmax(lm, __shfl_xor_sync(0xffffffffu, lm, off));
  for (int i = lane; i < n; i += 32) L.p[i] = exp((double)L.val[i] / T - lm);
  __syncwarp();
  double Z = 0.0;
  if (lane == 0)
    for (int i = 0; i < n; ++i) Z += L.p[i];
  Z = __shfl_sync(0xffffffffu, Z, 0);
  for (int i = lane; i < n; i += 32) L.p[i] = L.p[i] / Z;
  __syncwarp();
  if (!(top_p < 1.0)) return;

  // order by (logit desc, index asc): bitonic sort of a permutation
  int P2 = 1;
  while (P2 < n) P2 <<= 1;
  for (int i = lane; i < P2; i += 32) perm[i] = i < n ? i : -1;
  __syncwarp();
  for (int size = 2; size <= P2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = lane; i < P2; i += 32) {
        const int p = i ^ stride;
        if (p > i) {
          const bool asc = (i & size) == 0;
          const int a = perm[i], b = perm[p];
          bool a_first;
          if (a < 0) a_first = false;
          else if (b < 0) a_first = true;
          else a_first = (L.val[a] > L.val[b]) || (L.val[a] == L.val[b] && a < b);  // index order
          if (a_first != asc) {
            perm[i] = b;
            perm[p] = a;
          }
        }
      }
      __syncwarp();
    }
  }
  double S = 0.0;
  if (lane == 0) {
    double above = 0.0;
    int a = 0;
    while (a < n) {
      int b = a;
      while (b < n && L.val[perm[b]] == L.val[perm[a]]) ++b;
      const unsigned char kp = above < top_p ? 1 : 0;
      for (int c = a; c < b; ++c) keep[perm[c]] = kp;
      for (int c = a; c < b; ++c) above += L.p[perm[c]];
      a = b;
    }
    for (int i = 0; i < n; ++i)
      if (keep[i]) S += L.p[i];
  }
  __syncwarp();
  S = __shfl_sync(0xffffffffu, S, 0);
  for (int i = lane; i < n; i += 32) L.p[i] = keep[i] ? L.p[i] / S : 0.0;
  __syncwarp();
}

// Finish a row's candidate list: sort the buffer's first n entries by index
// (bitonic, padded to a power of two) and write count, indices and logits.
__device__ void finish_row(SelShared &s, int n, uint8_t *out) {
  const int tid = threadIdx.x;
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
  int *idxs = reinterpret_cast<int *>(out + 16);
  float *vals = reinterpret_cast<float *>(out + FINAL_V_OFF);
  for (int i = tid; i < n; i += SEL_THREADS) {
    idxs[i] = (int)s.idx[i];
    vals[i] = keyf(s.key[i]);
  }
  if (tid == 0) *reinterpret_cast<int *>(out) = n;
}


// Element e of this thread in the chunk starting at cb.  VEC: 16-byte loads
// (4 fp32 or 8 bf16 logits), the CTA's 256 loads of a step side by side.
template <typename T, bool VEC>
__device__ __forceinline__ long long sel_index(long long cb, int tid, int e) {
  if (!VEC) return cb + (long long)e * SEL_THREADS + tid;
  constexpr int PV = 16 / (int)sizeof(T);
  return cb + (long long)(e / PV) * (SEL_THREADS * PV) + (long long)tid * PV + (e % PV);
}

// This thread's SEL_PER_THREAD logits of the chunk at cb (0 past hi).
template <typename T, bool VEC>
__device__ __forceinline__ void sel_load(const T *z, long long cb, long long hi, int tid,
                                         float (&v)[SEL_PER_THREAD]) {
  if (!VEC) {
#pragma unroll
    for (int e = 0; e < SEL_PER_THREAD; ++e) {
      const long long i = sel_index<T, false>(cb, tid, e);
      v[e] = i < hi ? load_logit(z, i) : 0.f;
    }
    return;
  }
  constexpr int PV = 16 / (int)sizeof(T);
#pragma unroll
  for (int q = 0; q < SEL_PER_THREAD / PV; ++q) {
    const long long i0 = cb + (long long)q * (SEL_THREADS * PV) + (long long)tid * PV;
    if (i0 + PV <= hi) {
      const uint4 w = __ldcs(reinterpret_cast<const uint4 *>(z + i0));
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int x = 0; x < PV; ++x) {
        if (sizeof(T) == 4) v[q * PV + x] = __uint_as_float(u[x]);
        else v[q * PV + x] = __uint_as_float((x & 1) ? (u[x >> 1] & 0xFFFF0000u) : (u[x >> 1] << 16));
      }
    } else {
#pragma unroll
      for (int x = 0; x < PV; ++x) v[q * PV + x] = i0 + x < hi ? load_logit(z, i0 + x) : 0.f;
    }
  }
}

// One CTA per (row, chunk).  Streams the chunk once, keeping candidates above
// a running threshold; the exact top-k (with ties) of the chunk survives.
// With one chunk per row the list is written directly; otherwise the last
// CTA of the row to finish merges the chunk lists (the row's top-k is the
// top-k of the union of the chunks' top-k sets).
// Rows j in [jlo, jlo + jn) of every round (all 2K+1 rows, or only the draft
// rows when the target rows come from the lm_head's lists).
// VEC (rows on 16-byte boundaries): 16-byte loads.  Every thread keeps the
// next two steps' logits in flight while it filters the current one.
template <typename T, bool VEC>
__global__ void __launch_bounds__(SEL_THREADS, 4)
    select_kernel(const T *__restrict__ tgt, const T *__restrict__ drf, int K, int V, int k,
                  int C, int jlo, int jn, SelLayout lay, unsigned *err) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelShared &s = *reinterpret_cast<SelShared *>(smem_raw);
  __shared__ int s_last, s_off[MAX_CHUNKS + 1];
  const int tid = threadIdx.x, lane = tid & 31;
  const int rj = blockIdx.x / C, chunk = blockIdx.x % C;
  const int r = rj / jn, j = jlo + rj % jn;
  const int row = r * (2 * K + 1) + j;
  // (no early launch_dependents: the next stage is let in as this kernel's
  // CTAs exit; its small CTAs waiting beside this kernel slowed it)
  pdl_wait();
  const T *z = row_ptr(tgt, drf, r, j, K, V);
  // chunk bounds (multiples of the vector width with 16-byte loads)
  constexpr long long PV = VEC ? 16 / (long long)sizeof(T) : 1;
  const long long lo = (long long)chunk * V / C / PV * PV;
  const long long hi = chunk == C - 1 ? (long long)V : (long long)(chunk + 1) * V / C / PV * PV;
  if (tid == 0) {
    s.cnt = 0;
    s.tau = 0u;
  }
  __syncthreads();
  bool overflow = false;
  const int gap = imax(2 * k, 256);
  constexpr int SEL_ROOM = SEL_BUF - SEL_GROUP * SEL_CHUNK;  // kept entries a group can add to
  int trig = imin(SEL_ROOM, gap);
  int since = 0;  // chunks appended since the last barrier
  float vn[SEL_PER_THREAD], vnn[SEL_PER_THREAD];
  sel_load<T, VEC>(z, lo, hi, tid, vn);
  sel_load<T, VEC>(z, lo + SEL_CHUNK, hi, tid, vnn);
  for (long long cb = lo; cb < hi; cb += SEL_CHUNK) {
    const uint32_t tau = s.tau;
    float v[SEL_PER_THREAD];
#pragma unroll
    for (int e = 0; e < SEL_PER_THREAD; ++e) {
      v[e] = vn[e];
      vn[e] = vnn[e];
    }
    sel_load<T, VEC>(z, cb + 2 * SEL_CHUNK, hi, tid, vnn);
    // two chunks beyond the registers' prefetch on their way into L2 (16-byte
    // aligned rows only)
    if (VEC && tid == 0 && cb + SEL_PF * SEL_CHUNK < hi) {
      const long long c0 = cb + SEL_PF * SEL_CHUNK;
      const long long n = (hi - c0 < SEL_CHUNK ? hi - c0 : SEL_CHUNK) * (long long)sizeof(T) / 16 * 16;
      if (n > 0) l2_prefetch_bulk(z + c0, (uint32_t)n);
    }
    // The key order is the float order (logits are not NaN; keyf(fkey(x)) = x
    // with -0 taken as +0), so key >= tau iff the logit >= keyf(tau).  A lane
    // marks its passing logits; a warp with any appends them with one atomic
    // (offsets by a warp scan of the lanes' counts) and only the lanes that
    // hold candidates write.
    const float thr = tau == 0u ? -INFINITY : keyf(tau);
    float mx = v[0];
#pragma unroll
    for (int e = 1; e < SEL_PER_THREAD; ++e) mx = fmaxf(mx, v[e]);
    if (__any_sync(0xffffffffu, mx >= thr)) {
      unsigned pm = 0;
#pragma unroll
      for (int e = 0; e < SEL_PER_THREAD; ++e) pm |= (v[e] >= thr ? 1u : 0u) << e;
      if (cb + SEL_CHUNK > hi) {  // the range's last chunk: drop the padding past hi
#pragma unroll
        for (int e = 0; e < SEL_PER_THREAD; ++e)
          if (sel_index<T, VEC>(cb, tid, e) >= hi) pm &= ~(1u << e);
      }
      const int np = __popc(pm);
      int incl = np;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
      }
      int base = 0;
      if (lane == 31) base = atomicAdd(&s.cnt, incl);
      int pos = __shfl_sync(0xffffffffu, base, 31) + incl - np;
      if (pm) {
#pragma unroll
        for (int e = 0; e < SEL_PER_THREAD; ++e) {
          if (pm & (1u << e)) {
            s.key[pos] = fkey(v[e]);
            s.idx[pos] = (uint32_t)sel_index<T, VEC>(cb, tid, e);
            ++pos;
          }
        }
      }
    }
    // The CTA meets every SEL_GROUP chunks (the buffer holds that many
    // chunks beyond the trigger) and after its last chunk.  The threshold
    // changes only here.
    if (++since < SEL_GROUP && cb + SEL_CHUNK < hi) continue;
    since = 0;
    __syncthreads();  // every warp, whichever path it took
    // Compact (which raises the threshold to the buffer's k-th key) once the
    // buffer has gained max(2k, 256) candidates since the last compaction --
    // often enough that the threshold follows the row's top-k and few logits
    // pass -- and always before the next group of chunks could overflow it.
    if (s.cnt > trig) {
      compact(s, k);
      const int nc = s.cnt;
      __syncthreads();  // every thread has the count before any warp appends again
      if (nc > SEL_ROOM) {  // ties fill the buffer
        overflow = true;
        break;
      }
      trig = imin(SEL_ROOM, nc + gap);
    }
  }
  if (!overflow) compact(s, k);
  int n = s.cnt;
  overflow = overflow || n > CAND_MAX;
  if (C == 1) {
    uint8_t *out = lay.final + (size_t)row * ROW_BYTES;
    if (overflow) {
      if (tid == 0) {
        atomicOr(err, ERR_OVERFLOW);
        *reinterpret_cast<int *>(out) = -1;
      }
      return;
    }
    finish_row(s, n, out);
    return;
  }
  // ---- chunk list, then the last CTA of the row merges ----
  uint8_t *cl = lay.chunks + ((size_t)row * C + chunk) * ROW_BYTES;
  uint32_t *ckeys = reinterpret_cast<uint32_t *>(cl + 16);
  uint32_t *cidx = reinterpret_cast<uint32_t *>(cl + 16 + 4 * CAND_MAX);
  if (!overflow)
    for (int i = tid; i < n; i += SEL_THREADS) {
      ckeys[i] = s.key[i];
      cidx[i] = s.idx[i];
    }
  if (tid == 0) *reinterpret_cast<int *>(cl) = overflow ? -1 : n;
  __syncthreads();
  if (tid == 0) {
    // acquire-release arrival: the barrier before it puts the CTA's chunk
    // list ahead of the release, the barrier after it puts the merge's reads
    // behind the acquire
    unsigned prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(prev) : "l"(&lay.counters[row]) : "memory");
    s_last = prev == (unsigned)(C - 1);
    if (s_last) lay.counters[row] = 0u;  // ready for the next call
  }
  __syncthreads();
  if (!s_last) return;
  // chunk counts (one lane per chunk) and their prefix offsets
  if (tid < 32) {
    int c0 = -2, c1 = -2;  // -2: no such chunk
    if (tid < C) c0 = __ldcg(reinterpret_cast<const int *>(lay.chunks + ((size_t)row * C + tid) * ROW_BYTES));
    if (tid + 32 < C)
      c1 = __ldcg(reinterpret_cast<const int *>(lay.chunks + ((size_t)row * C + tid + 32) * ROW_BYTES));
    const bool bad = __any_sync(0xffffffffu, c0 == -1 || c1 == -1);
    int v0 = c0 > 0 ? c0 : 0, v1 = c1 > 0 ? c1 : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t0 = __shfl_up_sync(0xffffffffu, v0, off), t1 = __shfl_up_sync(0xffffffffu, v1, off);
      if (tid >= off) {
        v0 += t0;
        v1 += t1;
      }
    }
    const int tot0 = __shfl_sync(0xffffffffu, v0, 31);
    v1 += tot0;
    // inclusive sums -> exclusive offsets
    if (tid < C) s_off[tid] = v0 - (c0 > 0 ? c0 : 0);
    if (tid + 32 < C) s_off[tid + 32] = v1 - (c1 > 0 ? c1 : 0);
    const int total = __shfl_sync(0xffffffffu, v1, 31);
    if (tid == 0) s_off[C] = (bad || total > SEL_BUF) ? -1 : total;
  }
  __syncthreads();
  uint8_t *out = lay.final + (size_t)row * ROW_BYTES;
  const int total = s_off[C];
  if (total < 0) {
    if (tid == 0) {
      atomicOr(err, ERR_OVERFLOW);
      *reinterpret_cast<int *>(out) = -1;
    }
    return;
  }
  // gather every chunk's entries at once: entry e belongs to the last chunk
  // whose offset is <= e
  for (int e = tid; e < total; e += SEL_THREADS) {
    int lo = 0, hi = C - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_off[mid] <= e) lo = mid;
      else hi = mid - 1;
    }
    const uint8_t *src = lay.chunks + ((size_t)row * C + lo) * ROW_BYTES;
    const int i = e - s_off[lo];
    // asynchronous copies: every entry's load in flight at once
    cp_async4(&s.key[e], reinterpret_cast<const uint32_t *>(src + 16) + i);
    cp_async4(&s.idx[e], reinterpret_cast<const uint32_t *>(src + 16 + 4 * CAND_MAX) + i);
  }
  cp_async_wait_all();
  if (tid == 0) s.cnt = total;
  __syncthreads();
  compact(s, k);
  n = s.cnt;
  if (n > CAND_MAX) {
    if (tid == 0) {
      atomicOr(err, ERR_OVERFLOW);
      *reinterpret_cast<int *>(out) = -1;
    }
    return;
  }
  finish_row(s, n, out);
}

// The lm_head's lists (qmm_small_m_topk): a 64-byte header (rows M, CTAs,
// entries per list, k, vocabulary size) and per (lm_head row, CTA) a count
// then keys and indices of that CTA's top-k of its vocabulary range.
constexpr int LISTS_HDR = 64;
constexpr int MAX_LIST_CTAS = 1024;

// One CTA per target row (round r, row j <= K; lm_head row r*(K+1) + j): the
// union of the CTAs' lists reduced to the row's top-k (every logit equal to
// the k-th largest kept), written as the row's final list -- the result the
// select pass would give on the logits themselves.  When the lists fit the
// buffer together (the usual case: about k entries per CTA) every warp takes
// the top-k of its share of them and one warp the exact top-k of those
// candidates; otherwise they are compacted batch by batch.
constexpr int MERGE_WARPS = SEL_THREADS / 32;

// With draft lists (dlists non-null) every row of every round is merged --
// draft row i of round r is row r*K + i of the drafter's lm_head -- else only
// the target rows.
__global__ void __launch_bounds__(SEL_THREADS, 2)
    merge_lists_kernel(const uint8_t *__restrict__ tlists, const uint8_t *__restrict__ dlists,
                       int K, int k, SelLayout lay, unsigned *err) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  SelShared &s = *reinterpret_cast<SelShared *>(smem_raw);
  uint32_t *ckey = reinterpret_cast<uint32_t *>(smem_raw + sizeof(SelShared));  // [SEL_BUF]
  uint32_t *cidx = ckey + SEL_BUF;                                              // [SEL_BUF]
  __shared__ int s_off[MAX_LIST_CTAS + 1], s_cnt[MAX_LIST_CTAS];
  __shared__ int s_bad, s_c1, s_nc, s_wsum[MERGE_WARPS];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per_round = dlists ? 2 * K + 1 : K + 1;
  const int r = blockIdx.x / per_round, j = blockIdx.x % per_round;
  const int row = r * (2 * K + 1) + j;
  const uint8_t *lists = j <= K ? tlists : dlists;
  const int tr = j <= K ? r * (K + 1) + j : r * K + (j - K - 1);  // the lm_head's row
  pdl_wait();
  const int *hdr = reinterpret_cast<const int *>(lists);
  const int M = hdr[0], ctas = hdr[1], cap = hdr[2], klists = hdr[3];
  uint8_t *out = lay.final + (size_t)row * ROW_BYTES;
  // lists made for other rows or a smaller top-k cannot give this row's set
  if (tr >= M || klists < k || ctas < 1 || ctas > MAX_LIST_CTAS) {
    if (tid == 0) {
      atomicOr(err, ERR_LISTS);
      *reinterpret_cast<int *>(out) = -1;
    }
    return;
  }
  const size_t stride = 16 + (size_t)cap * 8;
  const uint8_t *base = lists + LISTS_HDR + (size_t)tr * ctas * stride;
  // every list's count, and their offsets (one block-wide exclusive scan)
  constexpr int PER = MAX_LIST_CTAS / SEL_THREADS;
  int c[PER], loc = 0;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int ci = tid * PER + e;
    c[e] = ci < ctas ? __ldcg(reinterpret_cast<const int *>(base + (size_t)ci * stride)) : 0;
    loc += c[e];
  }
  int incl = loc;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) s_wsum[warp] = incl;
  if (tid == 0) {
    s.cnt = 0;
    s_bad = 0;
  }
  __syncthreads();
  int wbase = 0, total = 0;
#pragma unroll
  for (int w = 0; w < MERGE_WARPS; ++w) {
    if (w < warp) wbase += s_wsum[w];
    total += s_wsum[w];
  }
  {
    int o = wbase + incl - loc;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int ci = tid * PER + e;
      if (ci < ctas) {
        s_cnt[ci] = c[e];
        s_off[ci] = o;
      }
      o += c[e];
    }
  }
  if (tid == 0) s_off[ctas] = total;
  __syncthreads();

  int n;
  if (total <= SEL_BUF) {
    // gather every list at once: entry e belongs to the last list whose
    // offset is <= e
    for (int e = tid; e < total; e += SEL_THREADS) {
      int lo = 0, hi = ctas - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_off[mid] <= e) lo = mid;
        else hi = mid - 1;
      }
      const uint8_t *src = base + (size_t)lo * stride;
      const int i = e - s_off[lo];
      cp_async4(&s.key[e], reinterpret_cast<const uint32_t *>(src + 16) + i);
      cp_async4(&s.idx[e], reinterpret_cast<const uint32_t *>(src + 16) + cap + i);
    }
    cp_async_wait_all();
    if (tid == 0) s_nc = 0;
    __syncthreads();
    // every warp: the top-k of its share, as candidates
    const int share = (total + MERGE_WARPS - 1) / MERGE_WARPS;
    const int a0 = imin(total, warp * share), a1 = imin(total, a0 + share);
    const uint32_t tw = warp_kth_largest(s.key + a0, a1 - a0, k);
    const unsigned lt = (1u << lane) - 1u;
    for (int b = a0; b < a1; b += 32) {
      const int i = b + lane;
      const bool keep = i < a1 && s.key[i] >= tw;
      const unsigned msk = __ballot_sync(0xffffffffu, keep);
      if (msk) {
        const int leader = __ffs(msk) - 1;
        int pos = 0;
        if (lane == leader) pos = atomicAdd(&s_nc, __popc(msk));
        pos = __shfl_sync(0xffffffffu, pos, leader) + __popc(msk & lt);
        if (keep) {
          ckey[pos] = s.key[i];
          cidx[pos] = s.idx[i];
        }
      }
    }
    __syncthreads();
    // one warp: the exact top-k of the candidates, back into the buffer
    if (warp == 0) {
      const int nc = s_nc;
      const uint32_t t = warp_kth_largest(ckey, nc, k);
      int w = 0;
      for (int b = 0; b < nc; b += 32) {
        const int i = b + lane;
        const bool keep = i < nc && ckey[i] >= t;
        const unsigned msk = __ballot_sync(0xffffffffu, keep);
        const int pos = w + __popc(msk & lt);
        if (keep && pos < SEL_BUF) {
          s.key[pos] = ckey[i];
          s.idx[pos] = cidx[i];
        }
        w += __popc(msk);
      }
      if (lane == 0) s.cnt = w;
    }
    __syncthreads();
    n = s.cnt;
  } else {
    // lists in batches whose entries fit the buffer beside the kept set
    for (int c0 = 0; c0 < ctas;) {
      int c1 = c0, tot = s.cnt;
      if (tid == 0) {
        while (c1 < ctas) {
          const int cn = s_cnt[c1];
          if (tot + cn > SEL_BUF) break;
          s_off[c1 - c0] = tot;
          tot += cn;
          ++c1;
        }
        s_off[c1 - c0] = tot;
        s_c1 = c1;
        if (c1 == c0) s_bad = 1;  // ties keep more than the buffer holds
      }
      __syncthreads();
      if (s_bad) break;
      c1 = s_c1;
      const int start = s.cnt, nb = c1 - c0;
      tot = s_off[nb];
      for (int e = start + tid; e < tot; e += SEL_THREADS) {
        int lo = 0, hi = nb - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (s_off[mid] <= e) lo = mid;
          else hi = mid - 1;
        }
        const uint8_t *src = base + (size_t)(c0 + lo) * stride;
        const int i = e - s_off[lo];
        cp_async4(&s.key[e], reinterpret_cast<const uint32_t *>(src + 16) + i);
        cp_async4(&s.idx[e], reinterpret_cast<const uint32_t *>(src + 16) + cap + i);
      }
      cp_async_wait_all();
      __syncthreads();
      if (tid == 0) s.cnt = tot;
      __syncthreads();
      compact(s, k);  // keeps the entries at or above the k-th largest key
      c0 = c1;
    }
    n = s.cnt;
  }
  if (s_bad || n > CAND_MAX) {
    if (tid == 0) {
      atomicOr(err, ERR_OVERFLOW);
      *reinterpret_cast<int *>(out) = -1;
    }
    return;
  }
  finish_row(s, n, out);
}

// One warp per candidate list: the truncated distribution, written beside
// the list (skipped for a list the select pass marked as overflowed).  Lists
// of up to DIST_SCAP entries are evaluated in shared memory; longer ones (a
// large top-k, or ties) in the row's own scratch space in global memory.
// Rows j in [jlo, jlo + jn) of every round; `rows` = R * jn.
__global__ void __launch_bounds__(DIST_WARPS * 32) dist_kernel(uint8_t *lists, int rows, int K,
                                                              int jlo, int jn, double temp,
                                                              double top_p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // (no early launch_dependents: the next stage is let in as this kernel's
  // CTAs exit; its small CTAs waiting beside this kernel slowed it)
  pdl_wait();
  const int rj = blockIdx.x * DIST_WARPS + warp;
  if (rj >= rows) return;
  const int row = (rj / jn) * (2 * K + 1) + jlo + rj % jn;
  uint8_t *in = lists + (size_t)row * ROW_BYTES;
  const int n = *reinterpret_cast<const int *>(in);
  if (n < 0) return;
  float *vsrc = reinterpret_cast<float *>(in + FINAL_V_OFF);
  double *pdst = reinterpret_cast<double *>(in + FINAL_P_OFF);
  if (n <= DIST_SCAP) {
    // per warp: probabilities, logits, sort permutation, keep flags
    uint8_t *ws = smem_raw + (size_t)warp * (DIST_SCAP * 17);
    double *p = reinterpret_cast<double *>(ws);
    float *val = reinterpret_cast<float *>(ws + 8 * DIST_SCAP);
    int *perm = reinterpret_cast<int *>(ws + 12 * DIST_SCAP);
    unsigned char *keep = ws + 16 * DIST_SCAP;
    for (int i = lane; i < n; i += 32) val[i] = vsrc[i];
    __syncwarp();
    List L{nullptr, val, p, n};
    dist(temp, top_p, L, perm, keep);
    for (int i = lane; i < n; i += 32) pdst[i] = p[i];
  } else {
    List L{nullptr, vsrc, pdst, n};
    dist(temp, top_p, L, reinterpret_cast<int *>(in + FINAL_PERM_OFF), in + FINAL_KEEP_OFF);
  }
}

// ------------------------------------------------------------- chain ---
struct ChainParams {
  const int32_t *drafts;
  const float *u;
  int32_t *out_tok, *out_n;
  const uint8_t *lists;  // select output [rows][ROW_BYTES]
  int R, K;
  unsigned *err;
};

// Load row (r, j)'s candidate list into L (index order): indices and the
// probabilities the dist kernel evaluated.  Returns the count, or -1 if the
// select pass overflowed.  Warp-cooperative.
__device__ int load_list(const ChainParams &cp, int r, int j, List &L) {
  const int lane = threadIdx.x;
  const uint8_t *in = cp.lists + ((size_t)r * (2 * cp.K + 1) + j) * ROW_BYTES;
  const int n = *reinterpret_cast<const int *>(in);
  if (n >= 0) {
    const int *idxs = reinterpret_cast<const int *>(in + 16);
    const double *ps = reinterpret_cast<const double *>(in + FINAL_P_OFF);
    for (int i = lane; i < n; i += 32) {
      L.idx[i] = idxs[i];
      L.p[i] = ps[i];
    }
  }
  __syncwarp();
  return n;
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

// One warp per round: the accept / residual / bonus chain on the
// distributions the dist kernel evaluated.
__global__ void __launch_bounds__(CHAIN_THREADS) chain_kernel(const ChainParams cp) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  double *pP = reinterpret_cast<double *>(smem_raw);
  double *pQ = pP + CAND_MAX;
  double *wv = pQ + CAND_MAX;
  int *iP = reinterpret_cast<int *>(wv + CAND_MAX);
  int *iQ = iP + CAND_MAX;

  const int r = blockIdx.x, lane = threadIdx.x;
  const int K = cp.K;
  pdl_launch_dependents();
  pdl_wait();
  List P{iP, nullptr, pP, 0}, Q{iQ, nullptr, pQ, 0};
  int32_t *tok = cp.out_tok + (size_t)r * (K + 1);
  const float *u = cp.u + (size_t)r * (K + 1);
  for (int i = lane; i <= K; i += 32) tok[i] = -1;
  __syncwarp();

  int n_acc = K;
  bool bad = false;  // a candidate list overflowed in the select pass
  for (int i = 0; i < K; ++i) {
    const int np = load_list(cp, r, i, P);
    const int nq = load_list(cp, r, K + 1 + i, Q);
    if (np < 0 || nq < 0) {
      bad = true;
      break;
    }
    P.n = np;
    Q.n = nq;
    int accept = 0;
    if (lane == 0) {
      const int x = cp.drafts[(size_t)r * K + i];
      const double px = lookup(P, x), qx = lookup(Q, x);
      accept = ((double)u[i] * qx < px) ? 1 : 0;
      if (accept) {
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
    accept = __shfl_sync(0xffffffffu, accept, 0);
    __syncwarp();
    if (!accept) {
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
      if (lane == 0) tok[K] = icdf(P, P.p, (double)u[K]);
    }
  }
  if (lane == 0) {
    if (bad) {
      cp.out_n[r] = -1;
      atomicOr(cp.err, ERR_OVERFLOW);
    } else {
      cp.out_n[r] = n_acc;
    }
  }
}

constexpr size_t CHAIN_SMEM = (size_t)CAND_MAX * (8 * 3 + 4 * 2);

// The select pass over rows j in [jlo, jlo + jn) of every round, with
// 16-byte loads when every row starts on a 16-byte boundary.
static cudaError_t launch_select(bool bf, const void *tgt, const void *drf, int K, int V, int k, int C,
                                 int jlo, int jn, SelLayout lay, unsigned *err, dim3 grid, size_t sm,
                                 cudaStream_t s) {
  const size_t esz = bf ? 2 : 4;
  const bool vec = (V * esz) % 16 == 0 && reinterpret_cast<uintptr_t>(tgt) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(drf) % 16 == 0;
  const dim3 b(SEL_THREADS);
  if (bf) {
    const auto *t = static_cast<const __nv_bfloat16 *>(tgt);
    const auto *d = static_cast<const __nv_bfloat16 *>(drf);
    return vec ? launch(select_kernel<__nv_bfloat16, true>, grid, b, sm, s, t, d, K, V, k, C, jlo, jn, lay, err)
               : launch(select_kernel<__nv_bfloat16, false>, grid, b, sm, s, t, d, K, V, k, C, jlo, jn, lay, err);
  }
  const auto *t = static_cast<const float *>(tgt);
  const auto *d = static_cast<const float *>(drf);
  return vec ? launch(select_kernel<float, true>, grid, b, sm, s, t, d, K, V, k, C, jlo, jn, lay, err)
             : launch(select_kernel<float, false>, grid, b, sm, s, t, d, K, V, k, C, jlo, jn, lay, err);
}

// Chunks per row the select pass may use: the most any k gives, over the
// rounds' 2K+1 rows (spec_accept) or their K draft rows alone
// (spec_accept_lists; fewer rows take more chunks each).
static int max_chunks(int R, int K, int V) {
  return chunks_per_row((long long)R * K, V, device_sm_count(), 0, SEL_BUF);
}

// Workspace of the candidate-list path: counters and final lists for every
// row, chunk lists for every row at the largest chunk count.
static size_t list_path_bytes(int R, int K, int V) {
  const long long rows = (long long)R * (2 * K + 1);
  return (sel_bytes(rows, max_chunks(R, K, V)) + 255) / 256 * 256;
}

}  // namespace acc
}  // namespace sv

using namespace sv;

extern "C" {

size_t spec_accept_workspace_bytes(int R, int K, int V) {
  if (R < 1 || K < 1 || V < 1) return 0;
  return acc::list_path_bytes(R, K, V) + acc::whole_workspace_bytes(R, K, V);
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
  const long long rows = (long long)R * (2 * K + 1);
  if (rows * acc::MAX_CHUNKS > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < spec_accept_workspace_bytes(R, K, V)) return SV_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t list_bytes = acc::list_path_bytes(R, K, V);
  const bool top_k_on = params.top_k > 0 && params.top_k < V;
  if (T > 0.f && !(top_k_on && params.top_k <= acc::MAX_TOPK)) {
    // top-k off or beyond the candidate lists: the whole-vocabulary path
    acc::WholeArgs a{};
    a.tgt = target_logits;
    a.drf = draft_logits;
    a.bf16 = logit_dtype == SV_BF16;
    a.drafts = draft_tokens;
    a.u = uniforms;
    a.out_tok = out_tokens;
    a.out_n = out_num_accepted;
    a.R = R;
    a.K = K;
    a.V = V;
    a.temperature = T;
    a.top_k = top_k_on ? params.top_k : 0;
    a.top_p = tp;
    a.workspace = static_cast<uint8_t *>(workspace) + list_bytes;
    a.ws_bytes = ws_bytes - list_bytes;
    return acc::whole_launch(a, s);
  }
  const int k = T == 0.f ? 1 : params.top_k;
  const int C = acc::chunks_per_row(rows, V, device_sm_count(), k, acc::SEL_BUF);
  unsigned *err = device_error_word();
  if (!err) return SV_ERR_CUDA;
  const int bf = logit_dtype == SV_BF16;
  cudaError_t e = cudaSuccess;
  acc::SelLayout lay{};
  uint8_t *w = static_cast<uint8_t *>(workspace);
  lay.counters = reinterpret_cast<unsigned *>(w);
  lay.final = w + ((size_t)rows * 4 + 255) / 256 * 256;
  lay.chunks = lay.final + (size_t)rows * acc::ROW_BYTES;
  const size_t sm = sizeof(acc::SelShared);
  const dim3 grid((unsigned)(rows * C));
  e = acc::launch_select(bf, target_logits, draft_logits, K, V, k, C, 0, 2 * K + 1, lay, err, grid, sm, s);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  e = launch(acc::dist_kernel, dim3((unsigned)((rows + acc::DIST_WARPS - 1) / acc::DIST_WARPS)),
             dim3(acc::DIST_WARPS * 32), (size_t)acc::DIST_WARPS * acc::DIST_SCAP * 17, s, lay.final,
             (int)rows, K, 0, 2 * K + 1, (double)T, (double)tp);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  acc::ChainParams cp{};
  cp.drafts = draft_tokens;
  cp.u = uniforms;
  cp.out_tok = out_tokens;
  cp.out_n = out_num_accepted;
  cp.lists = lay.final;
  cp.R = R;
  cp.K = K;
  cp.err = err;
  e = launch(acc::chain_kernel, dim3(R), dim3(acc::CHAIN_THREADS), acc::CHAIN_SMEM, s, cp);
  return from_cuda(e);
}

// The candidate-list settings (temperature 0, or 0 < top_k <= 1024 below V);
// the host checks shared by the two calls below.  Returns the top-k or a
// negative status.
static int lists_k(sv_sampling_params params, int R, int K, int V, void *workspace,
                   size_t ws_bytes) {
  if (R < 1 || K < 1 || V < 1) return -SV_ERR_INVALID_ARG;
  const float T = params.temperature, tp = params.top_p;
  if (!(T >= 0.f) || !(T < INFINITY)) return -SV_ERR_INVALID_ARG;
  if (!(tp > 0.f && tp <= 1.f)) return -SV_ERR_INVALID_ARG;
  if (params.top_k < 0) return -SV_ERR_INVALID_ARG;
  if (K > acc::MAX_K) return -SV_ERR_UNSUPPORTED;
  if (T > 0.f && !(params.top_k > 0 && params.top_k < V && params.top_k <= acc::MAX_TOPK))
    return -SV_ERR_UNSUPPORTED;
  const long long rows = (long long)R * (2 * K + 1);
  if (rows * acc::MAX_CHUNKS > 0x7fffffffLL) return -SV_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < spec_accept_workspace_bytes(R, K, V)) return -SV_ERR_WORKSPACE;
  return T == 0.f ? 1 : params.top_k;
}

static acc::SelLayout lists_layout(void *workspace, int R, int K) {
  const long long rows = (long long)R * (2 * K + 1);
  acc::SelLayout lay{};
  uint8_t *w = static_cast<uint8_t *>(workspace);
  lay.counters = reinterpret_cast<unsigned *>(w);
  lay.final = w + ((size_t)rows * 4 + 255) / 256 * 256;
  lay.chunks = lay.final + (size_t)rows * acc::ROW_BYTES;
  return lay;
}

sv_status spec_accept_draft_select(const void *draft_logits, sv_dtype logit_dtype,
                                   sv_sampling_params params, int R, int K, int V, void *workspace,
                                   size_t ws_bytes, sv_stream_t stream) {
  if (!draft_logits) return SV_ERR_INVALID_ARG;
  if (logit_dtype != SV_F32 && logit_dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  const int k = lists_k(params, R, K, V, workspace, ws_bytes);
  if (k < 0) return (sv_status)-k;
  const int C = acc::chunks_per_row((long long)R * K, V, device_sm_count(), k, acc::SEL_BUF);
  unsigned *err = device_error_word();
  if (!err) return SV_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const acc::SelLayout lay = lists_layout(workspace, R, K);
  const size_t sm = sizeof(acc::SelShared);
  const dim3 grid((unsigned)((long long)R * K * C));
  cudaError_t e = acc::launch_select(logit_dtype == SV_BF16, nullptr, draft_logits, K, V, k, C, K + 1, K,
                                     lay, err, grid, sm, s);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  const int drows = R * K;
  e = launch(acc::dist_kernel, dim3((unsigned)((drows + acc::DIST_WARPS - 1) / acc::DIST_WARPS)),
             dim3(acc::DIST_WARPS * 32), (size_t)acc::DIST_WARPS * acc::DIST_SCAP * 17, s, lay.final,
             drows, K, K + 1, K, (double)params.temperature, (double)params.top_p);
  return from_cuda(e);
}

sv_status spec_accept_lists(const void *target_lists, const void *draft_lists,
                            const int32_t *draft_tokens, const float *uniforms,
                            sv_sampling_params params, int R, int K, int V, int32_t *out_tokens,
                            int32_t *out_num_accepted, void *workspace, size_t ws_bytes,
                            sv_stream_t stream) {
  if (!target_lists || !draft_tokens || !uniforms || !out_tokens || !out_num_accepted)
    return SV_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(target_lists) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(draft_lists) % 16 != 0)
    return SV_ERR_INVALID_ARG;
  const int k = lists_k(params, R, K, V, workspace, ws_bytes);
  if (k < 0) return (sv_status)-k;
  unsigned *err = device_error_word();
  if (!err) return SV_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const acc::SelLayout lay = lists_layout(workspace, R, K);
  const size_t sm = sizeof(acc::SelShared);
  cudaError_t e;
  // the target rows, and the draft rows too when their lists are given
  const int jn = draft_lists ? 2 * K + 1 : K + 1;
  const int mrows = R * jn;
  e = launch(acc::merge_lists_kernel, dim3((unsigned)mrows), dim3(acc::SEL_THREADS),
             sm + (size_t)acc::SEL_BUF * 8, s, static_cast<const uint8_t *>(target_lists),
             static_cast<const uint8_t *>(draft_lists), K, k, lay, err);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  e = launch(acc::dist_kernel, dim3((unsigned)((mrows + acc::DIST_WARPS - 1) / acc::DIST_WARPS)),
             dim3(acc::DIST_WARPS * 32), (size_t)acc::DIST_WARPS * acc::DIST_SCAP * 17, s, lay.final,
             mrows, K, 0, jn, (double)params.temperature, (double)params.top_p);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  acc::ChainParams cp{};
  cp.drafts = draft_tokens;
  cp.u = uniforms;
  cp.out_tok = out_tokens;
  cp.out_n = out_num_accepted;
  cp.lists = lay.final;
  cp.R = R;
  cp.K = K;
  cp.err = err;
  e = launch(acc::chain_kernel, dim3(R), dim3(acc::CHAIN_THREADS), acc::CHAIN_SMEM, s, cp);
  return from_cuda(e);
}

}  // extern "C"
