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
// and v[i]), so one warp owns one row for the whole call: the row sits in
// registers (dk/32 floats a lane), each token costs two warp all-reduces (S k
// and S q) and one fused update, and the committed row is written back once.
// Eight warps of a CTA take eight consecutive rows, so they read the same key
// and query vectors (from L1 after the first).  Bound by HBM (state read +
// write) at these sizes, and by the per-token dependency chain at small ones.
#include "common.cuh"

namespace sv {
namespace gdn {

constexpr int WARPS = 8;

template <int CPL>
__device__ __forceinline__ void load_bf16(const __nv_bfloat16 *p, float (&x)[CPL]) {
  if constexpr (CPL == 2) {
    const uint32_t w = *reinterpret_cast<const uint32_t *>(p);
    x[0] = bf16lo(w);
    x[1] = bf16hi(w);
  } else if constexpr (CPL == 4) {
    const uint2 w = *reinterpret_cast<const uint2 *>(p);
    x[0] = bf16lo(w.x), x[1] = bf16hi(w.x), x[2] = bf16lo(w.y), x[3] = bf16hi(w.y);
  } else {
    const uint4 w = *reinterpret_cast<const uint4 *>(p);
    x[0] = bf16lo(w.x), x[1] = bf16hi(w.x), x[2] = bf16lo(w.y), x[3] = bf16hi(w.y);
    x[4] = bf16lo(w.z), x[5] = bf16hi(w.z), x[6] = bf16lo(w.w), x[7] = bf16hi(w.w);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

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

// One token of the rule on this lane's CPL columns of row i; returns S k.
template <int CPL>
__device__ __forceinline__ void step(float (&row)[CPL], const float (&kk)[CPL], float vi, float a,
                                     float bb) {
  float u = 0.f;
#pragma unroll
  for (int c = 0; c < CPL; ++c) u = fmaf(row[c], kk[c], u);
  u = warp_sum(u);
  const float coef = bb * (vi - a * u);
#pragma unroll
  for (int c = 0; c < CPL; ++c) row[c] = fmaf(a, row[c], coef * kk[c]);
}

template <int DK>
__global__ void __launch_bounds__(WARPS * 32) gdn_kernel(const Params P) {
  constexpr int CPL = DK / 32;  // columns a lane holds
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (w >= (long long)P.Hv * P.dv) return;
  const int h = (int)(w / P.dv), i = (int)(w % P.dv);
  const int hk = h / (P.Hv / P.Hk);
  float *srow = P.state + (size_t)w * DK + lane * CPL;
  float row[CPL];
#pragma unroll
  for (int c = 0; c < CPL; c += 2) {
    const float2 x = *reinterpret_cast<const float2 *>(srow + c);
    row[c] = x.x;
    row[c + 1] = x.y;
  }
  // commit: the accepted prefix of the previous round
  for (int t = 0; t < P.n_replay; ++t) {
    float kk[CPL];
    load_bf16<CPL>(P.tk + ((size_t)t * P.Hk + hk) * DK + lane * CPL, kk);
    const float vi = __bfloat162float(P.tv[((size_t)t * P.Hv + h) * P.dv + i]);
    step<CPL>(row, kk, vi, expf(P.tg[(size_t)t * P.Hv + h]), P.tb[(size_t)t * P.Hv + h]);
  }
  if (P.n_replay > 0) {
#pragma unroll
    for (int c = 0; c < CPL; c += 2) *reinterpret_cast<float2 *>(srow + c) = make_float2(row[c], row[c + 1]);
  }
  // this round's rows, from the committed state (kept in registers only)
  for (int t = 0; t < P.M; ++t) {
    float kk[CPL], qq[CPL];
    load_bf16<CPL>(P.k + ((size_t)t * P.Hk + hk) * DK + lane * CPL, kk);
    load_bf16<CPL>(P.q + ((size_t)t * P.Hk + hk) * DK + lane * CPL, qq);
    const float vi = __bfloat162float(P.v[((size_t)t * P.Hv + h) * P.dv + i]);
    step<CPL>(row, kk, vi, expf(P.g[(size_t)t * P.Hv + h]), P.b[(size_t)t * P.Hv + h]);
    float ov = 0.f;
#pragma unroll
    for (int c = 0; c < CPL; ++c) ov = fmaf(row[c], qq[c], ov);
    ov = warp_sum(ov);
    if (lane == 0) {
      const size_t oi = ((size_t)t * P.Hv + h) * P.dv + i;
      if (P.o_f32)
        static_cast<float *>(P.o)[oi] = ov;
      else
        static_cast<__nv_bfloat16 *>(P.o)[oi] = __float2bfloat16_rn(ov);
    }
  }
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
  const long long rows = (long long)Hv * dv;
  const long long blocks = (rows + gdn::WARPS - 1) / gdn::WARPS;
  if (blocks > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
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
  const dim3 grid((unsigned)blocks), block(gdn::WARPS * 32);
  cudaError_t e;
  switch (dk) {
    case 64: e = launch(gdn::gdn_kernel<64>, grid, block, 0, s, P); break;
    case 128: e = launch(gdn::gdn_kernel<128>, grid, block, 0, s, P); break;
    default: e = launch(gdn::gdn_kernel<256>, grid, block, 0, s, P); break;
  }
  return from_cuda(e);
}

}  // extern "C"
