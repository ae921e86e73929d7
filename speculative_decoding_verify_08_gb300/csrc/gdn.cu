// gdn.cu -- GatedDeltaNet verify step with deferred commit (tape replay).
//
// Most layers of the hybrid targets are GatedDeltaNet layers whose recurrent
// state is a fixed-size array: a rejected draft cannot be trimmed from it the
// way a KV cache is truncated, and MTPLX rolls it back by replaying an
// "innovation tape" in its GDN kernel ("Speculative decoding and MTP on Apple
// silicon", Facts).  Per value head h (key head g = h / (Hv/Hk)) the state S
// is dv x dk and every token applies the gated delta rule
//     S <- a S (I - b k k^T) + b v k^T = a S + b (v - a S k) k^T,  a = exp(g),
// and reads o = S q.  A verify round runs its M rows from the committed state
// without writing it; the next call first replays the accepted prefix of that
// round (its own k, v, g, b: the tape) into the state, once acceptance is
// known.  The state is therefore read once and written once per round.
//
// Design: rows of S are independent under the rule (row i needs only S[i,:]
// and v[i]), so each row stays in registers for the whole call; the call is a
// chain of dependent per-token steps (dot product, reduction, update), so
// what bounds it is that chain's latency and instruction count.  Eight lanes
// share a row (three-step shuffle reductions), a lane holding four-column
// pieces 32 columns apart so that the row's lanes read one contiguous
// 128-byte line of a key per piece (no bank conflicts) and keep four
// independent partial sums; a 64-thread CTA holds eight rows of one value
// head (many small CTAs spread evenly over the SMs) and first stages every
// token's key, query, value and gates of that head in shared memory (fp32).
// The committed rows are written back once.  The successor kernel is let in
// only at the end: its CTAs waiting beside this latency-bound chain slowed
// it by a third.
#include "common.cuh"

namespace sv {
namespace gdn {

constexpr int WARPS = 2;
constexpr int LPR = 8;                  // lanes per state row
constexpr int ROWS = WARPS * 32 / LPR;  // rows per CTA (8)
constexpr int MAX_TOKENS = 64;          // per call, for each of replay and verify
constexpr int STAGE_U = 4;              // key and query pieces a thread loads per round
constexpr int STAGE_V = 2;              // value items a thread loads ahead

struct Params {
  float *state;  // [Hv][dv][dk]
  const __nv_bfloat16 *tk, *tv;
  const float *tg, *tb;
  int n_replay;
  const __nv_bfloat16 *q, *k, *v;
  const float *g, *b;
  void *o;
  int o_f32;
  int M, Hk, Hv, dv;
};

__host__ __device__ inline size_t smem_bytes(int DK, int T, int M) {
  return ((size_t)T * DK + (size_t)M * DK + (size_t)T * ROWS + 2 * (size_t)T) * sizeof(float);
}

// lane `sub` of a row holds columns sub*4 + 32*j .. +3 (j < DK/32): the eight
// lanes of a row read one contiguous 128-byte line of a key per j
template <int NJ>
__device__ __forceinline__ float dot_strided(const float (&row)[NJ * 4], const float *x) {
  float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int jj = 0; jj < NJ; ++jj) {
    const float4 x4 = *reinterpret_cast<const float4 *>(x + 32 * jj);
    s[0] = fmaf(row[4 * jj], x4.x, s[0]);
    s[1] = fmaf(row[4 * jj + 1], x4.y, s[1]);
    s[2] = fmaf(row[4 * jj + 2], x4.z, s[2]);
    s[3] = fmaf(row[4 * jj + 3], x4.w, s[3]);
  }
  return (s[0] + s[1]) + (s[2] + s[3]);
}

__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

template <int DK>
__global__ void __launch_bounds__(WARPS * 32) gdn_kernel(const Params P) {
  constexpr int NJ = DK / 32;  // float4 chunks a lane holds
  constexpr int CPL = NJ * 4;
  extern __shared__ __align__(16) float sm[];
  const int T = P.n_replay + P.M;
  float *sk = sm, *sq = sk + (size_t)T * DK, *sv_ = sq + (size_t)P.M * DK, *sab = sv_ + (size_t)T * ROWS;
  const int h = blockIdx.y, i0 = blockIdx.x * ROWS;
  const int hk = h / (P.Hv / P.Hk);
  const int tid = threadIdx.x, lane = tid & 31;
  const int r = tid / LPR, sub = lane % LPR;
  const int i = i0 + r;
  const bool live = i < P.dv;
  pdl_wait();
  float *srow = P.state + ((size_t)h * P.dv + (live ? i : 0)) * DK + sub * 4;
  float row[CPL];
#pragma unroll
  for (int jj = 0; jj < NJ; ++jj) {
    const float4 x = live ? *reinterpret_cast<const float4 *>(srow + 32 * jj) : make_float4(0.f, 0.f, 0.f, 0.f);
    row[4 * jj] = x.x, row[4 * jj + 1] = x.y, row[4 * jj + 2] = x.z, row[4 * jj + 3] = x.w;
  }
  // Staging, each thread's global loads issued before its shared stores (a
  // loop that loads and stores in turn waits for memory once per item): the
  // first values and gates into registers, the keys and queries in rounds of
  // STAGE_U 16-byte pieces per thread, then the values and gates stored.
  constexpr int NT = WARPS * 32;
  const int n = P.n_replay;
  auto vload = [&](int e) -> float {
    const int t = e / ROWS, rr = e % ROWS;
    if (i0 + rr >= P.dv) return 0.f;
    return __bfloat162float(t < n ? P.tv[((size_t)t * P.Hv + h) * P.dv + i0 + rr]
                                  : P.v[((size_t)(t - n) * P.Hv + h) * P.dv + i0 + rr]);
  };
  auto gload = [&](int t, float &gv, float &bv) {
    const size_t gi = (size_t)(t < n ? t : t - n) * P.Hv + h;
    gv = t < n ? P.tg[gi] : P.g[gi];
    bv = t < n ? P.tb[gi] : P.b[gi];
  };
  float vreg[STAGE_V], greg = 0.f, breg = 0.f;
#pragma unroll
  for (int u = 0; u < STAGE_V; ++u) vreg[u] = tid + u * NT < T * ROWS ? vload(tid + u * NT) : 0.f;
  if (tid < T) gload(tid, greg, breg);
  // pieces e < T * DK / 8 are keys (token e / (DK / 8)), the rest queries;
  // the queries' rows follow the keys' in shared memory
  const int nkq = (T + P.M) * (DK / 8);
  for (int base = 0; base < nkq; base += STAGE_U * NT) {
    uint4 w[STAGE_U];
#pragma unroll
    for (int u = 0; u < STAGE_U; ++u) {
      const int e = base + u * NT + tid;
      if (e < nkq) {
        const int t = e / (DK / 8), c8 = e % (DK / 8);
        const __nv_bfloat16 *src = t < n   ? P.tk + ((size_t)t * P.Hk + hk) * DK
                                   : t < T ? P.k + ((size_t)(t - n) * P.Hk + hk) * DK
                                           : P.q + ((size_t)(t - T) * P.Hk + hk) * DK;
        w[u] = *reinterpret_cast<const uint4 *>(src + c8 * 8);
      }
    }
#pragma unroll
    for (int u = 0; u < STAGE_U; ++u) {
      const int e = base + u * NT + tid;
      if (e < nkq) {
        float4 *d = reinterpret_cast<float4 *>(sk + (size_t)e * 8);
        d[0] = make_float4(bf16lo(w[u].x), bf16hi(w[u].x), bf16lo(w[u].y), bf16hi(w[u].y));
        d[1] = make_float4(bf16lo(w[u].z), bf16hi(w[u].z), bf16lo(w[u].w), bf16hi(w[u].w));
      }
    }
  }
#pragma unroll
  for (int u = 0; u < STAGE_V; ++u)
    if (tid + u * NT < T * ROWS) sv_[tid + u * NT] = vreg[u];
  for (int e = tid + STAGE_V * NT; e < T * ROWS; e += NT) sv_[e] = vload(e);
  if (tid < T) {
    sab[2 * tid] = expf(greg);
    sab[2 * tid + 1] = breg;
  }
  for (int t = tid + NT; t < T; t += NT) {
    float gv, bv;
    gload(t, gv, bv);
    sab[2 * t] = expf(gv);
    sab[2 * t + 1] = bv;
  }
  __syncthreads();

  for (int t = 0; t < T; ++t) {
    if (t == P.n_replay && P.n_replay > 0 && live) {
#pragma unroll
      for (int jj = 0; jj < NJ; ++jj)
        *reinterpret_cast<float4 *>(srow + 32 * jj) =
            make_float4(row[4 * jj], row[4 * jj + 1], row[4 * jj + 2], row[4 * jj + 3]);
    }
    const float *kk = sk + (size_t)t * DK + sub * 4;
    const float u = row_sum(dot_strided<NJ>(row, kk));
    const float a = sab[2 * t];
    const float coef = sab[2 * t + 1] * (sv_[t * ROWS + r] - a * u);
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
      const float4 k4 = *reinterpret_cast<const float4 *>(kk + 32 * jj);
      row[4 * jj] = fmaf(a, row[4 * jj], coef * k4.x);
      row[4 * jj + 1] = fmaf(a, row[4 * jj + 1], coef * k4.y);
      row[4 * jj + 2] = fmaf(a, row[4 * jj + 2], coef * k4.z);
      row[4 * jj + 3] = fmaf(a, row[4 * jj + 3], coef * k4.w);
    }
    if (t >= P.n_replay) {
      const int tv = t - P.n_replay;
      const float ov = row_sum(dot_strided<NJ>(row, sq + (size_t)tv * DK + sub * 4));
      if (sub == 0 && live) {
        const size_t oi = ((size_t)tv * P.Hv + h) * P.dv + i;
        if (P.o_f32)
          static_cast<float *>(P.o)[oi] = ov;
        else
          static_cast<__nv_bfloat16 *>(P.o)[oi] = __float2bfloat16_rn(ov);
      }
    }
  }
  if (P.M == 0 && P.n_replay > 0 && live) {
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj)
      *reinterpret_cast<float4 *>(srow + 32 * jj) =
          make_float4(row[4 * jj], row[4 * jj + 1], row[4 * jj + 2], row[4 * jj + 3]);
  }
  // the successor is let in only now: its waiting CTAs would otherwise share
  // the SMs with this kernel's latency-bound token chain
  pdl_launch_dependents();
}

}  // namespace gdn
}  // namespace sv

using namespace sv;

extern "C" {

sv_status gdn_verify(float *state, const void *tape_k, const void *tape_v, const float *tape_g,
                     const float *tape_beta, int n_replay, const void *q, const void *k,
                     const void *v, const float *g, const float *beta, void *o, sv_dtype o_dtype,
                     int M, int Hk, int Hv, int dk, int dv, sv_stream_t stream) {
  if (!state || M < 0 || n_replay < 0 || M + n_replay < 1) return SV_ERR_INVALID_ARG;
  if (Hk < 1 || Hv < 1 || Hv % Hk != 0 || dv < 1) return SV_ERR_INVALID_ARG;
  if (dk != 64 && dk != 128 && dk != 256) return SV_ERR_UNSUPPORTED;
  if (o_dtype != SV_BF16 && o_dtype != SV_F32) return SV_ERR_INVALID_ARG;
  if (n_replay > 0 && (!tape_k || !tape_v || !tape_g || !tape_beta)) return SV_ERR_INVALID_ARG;
  if (M > 0 && (!q || !k || !v || !g || !beta || !o)) return SV_ERR_INVALID_ARG;
  for (const void *p : {(const void *)state, tape_k, q, k})
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return SV_ERR_INVALID_ARG;
  if (n_replay > gdn::MAX_TOKENS || M > gdn::MAX_TOKENS) return SV_ERR_UNSUPPORTED;
  if (Hv > 65535) return SV_ERR_UNSUPPORTED;
  gdn::Params P{};
  P.state = state;
  P.tk = static_cast<const __nv_bfloat16 *>(tape_k);
  P.tv = static_cast<const __nv_bfloat16 *>(tape_v);
  P.tg = tape_g;
  P.tb = tape_beta;
  P.n_replay = n_replay;
  P.q = static_cast<const __nv_bfloat16 *>(q);
  P.k = static_cast<const __nv_bfloat16 *>(k);
  P.v = static_cast<const __nv_bfloat16 *>(v);
  P.g = g;
  P.b = beta;
  P.o = o;
  P.o_f32 = o_dtype == SV_F32 ? 1 : 0;
  P.M = M;
  P.Hk = Hk;
  P.Hv = Hv;
  P.dv = dv;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const dim3 grid((unsigned)((dv + gdn::ROWS - 1) / gdn::ROWS), (unsigned)Hv), block(gdn::WARPS * 32);
  const size_t smem = gdn::smem_bytes(dk, n_replay + M, M);
  cudaError_t e;
  switch (dk) {
    case 64: e = launch(gdn::gdn_kernel<64>, grid, block, smem, s, P); break;
    case 128: e = launch(gdn::gdn_kernel<128>, grid, block, smem, s, P); break;
    default: e = launch(gdn::gdn_kernel<256>, grid, block, smem, s, P); break;
  }
  return from_cuda(e);
}

}  // extern "C"
