// qmm.cu -- small-M matmul over 4-bit affine group-quantised weights.
//
//   y[m][n] = sum_k x[m][k] * (s[n][g] * q[n][k] + b[n][g]),  g = k / 64
//
// The verify pass multiplies M = K+1 <= 16 activation rows by every weight
// matrix of the model, so the kernel is bound by reading the weights once
// ("The fastest way to run local LLMs on a Mac", "Decode is a memory-bandwidth
// problem"; "Speculative decoding and MTP on Apple silicon", Facts: the stock
// quantized matmul re-reads the weights per row for M = 2..8, a small-M kernel
// shares them across up to 16 rows).
//
// Design (GB300):
//  * Weights are prepacked once into 16-row x 64-k blocks of 576 bytes: the
//    512 code bytes are laid out so that lane L of a warp reads its 16 bytes
//    and holds, per k16 step, exactly the A fragment of an m16n8k16 MMA for
//    8 codes; the 64 trailing bytes hold that block's 16 scales and biases.
//  * Per CTA (one per SM), a producer warp streams contiguous runs of blocks
//    with TMA bulk copies (cp.async.bulk, L2 evict-first) into a 24-stage
//    shared-memory ring; eight consumer warps each own one 16-row tile.
//  * Dequantisation is one LOP3 per pair of codes: (code | 0x4300) is the
//    bf16 value 128 + code, exact.  The MMA computes sum_k x*(128+q) per
//    group in fp32; the affine terms are folded per group:
//       sum_k x*(s*q + b) = s * acc + (b - 128*s) * sum_k x.
//  * Activations are staged once per K slice into shared memory in fragment
//    order together with their per-group sums.  M <= 8 uses one n8 half of
//    the MMA, M <= 16 two halves; the weight fragment is shared by both.
//  * K is split into slices of at most 40 groups when that balances the SMs
//    better (plan depends on N, K and the SM count only, never on M); the
//    last warp to finish a tile sums the slice partials in slice order.
#include <algorithm>

#include "common.cuh"

namespace sv {
namespace qmm {

constexpr int TILE_N = 16;
constexpr int GROUP = 64;
constexpr int BLOCK_BYTES = 576;   // 512 B codes + 64 B scales/biases
constexpr int CODE_BYTES = 512;
constexpr int KB_GROUPS = 8;       // groups per pipeline stage
constexpr int STAGE_BYTES = KB_GROUPS * BLOCK_BYTES;
constexpr int NSTAGE = 24;
constexpr int CWARPS = 8;          // consumer warps
constexpr int THREADS = (CWARPS + 1) * 32;
constexpr int MAX_SLICE_GROUPS = 40;
constexpr int BAR_BYTES = 1024;

struct Plan {
  int NT;     // 16-row tiles
  int G;      // groups per row
  int S;      // K slices
  int GS;     // groups per slice (the last may be shorter)
  int units;  // S * NT (slice-major)
  int ctas;   // grid size
};

static Plan make_plan(int N, int K, int sms) {
  Plan p{};
  p.NT = (N + TILE_N - 1) / TILE_N;
  p.G = K / GROUP;
  const int smin = (p.G + MAX_SLICE_GROUPS - 1) / MAX_SLICE_GROUPS;
  double best = 1e300;
  for (int S = smin; S <= p.G && S <= 64; ++S) {
    const int GS = (p.G + S - 1) / S;
    const int Se = (p.G + GS - 1) / GS;
    if (Se != S) continue;  // every slice non-empty
    const long long units = (long long)S * p.NT;
    const int ctas = (int)std::min<long long>(units, sms);
    const long long per = (units + ctas - 1) / ctas;
    // bytes on the busiest SM, plus one block's worth per split partial
    const double cost = (double)per * GS + (S > 1 ? (double)per : 0.0);
    if (cost < best - 1e-9) {
      best = cost;
      p.S = S;
      p.GS = GS;
      p.units = (int)units;
      p.ctas = ctas;
    }
  }
  return p;
}

static size_t smem_bytes(int H) {
  return BAR_BYTES + (size_t)NSTAGE * STAGE_BYTES + (size_t)MAX_SLICE_GROUPS * H * 1024 +
         (size_t)MAX_SLICE_GROUPS * 16 * sizeof(float);
}

static size_t workspace_bytes(const Plan &p) {
  if (p.S <= 1) return 0;
  const size_t counters = ((size_t)p.NT * 4 + 255) / 256 * 256;
  return counters + (size_t)p.S * p.NT * 32 * 8 * sizeof(float);
}

// ----------------------------------------------------------- prepack ---
// One thread per (tile, group, lane): gathers the 32 codes lane `lane` needs
// for the four k16 steps of the group.  Nibble j of step word s holds
//   row gq + 8*(j&1), k = 16s + 2tq + 8*((j>>1)&1) + ((j>>2)&1)
// so that (w >> 4i) & 0x000F000F yields MMA A-fragment register i.
__global__ void prepack_kernel(const uint32_t *__restrict__ wq, const uint16_t *__restrict__ sc,
                               const uint16_t *__restrict__ bi, int N, int K, int NT, int G,
                               uint8_t *__restrict__ out) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)NT * G * 32) return;
  const int lane = (int)(idx & 31);
  const long long tg = idx >> 5;
  const int g = (int)(tg % G);
  const int t = (int)(tg / G);
  const int gq = lane >> 2, tq = lane & 3;
  const int KW = K / 8;
  uint32_t words[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int row = gq + ((j & 1) ? 8 : 0);
      const int kk = 16 * s + 2 * tq + ((j & 2) ? 8 : 0) + ((j & 4) ? 1 : 0);
      const int n = TILE_N * t + row;
      const int k = GROUP * g + kk;
      uint32_t code = 0;
      if (n < N) code = (wq[(size_t)n * KW + (k >> 3)] >> (4 * (k & 7))) & 15u;
      w |= code << (4 * j);
    }
    words[s] = w;
  }
  uint8_t *blk = out + ((size_t)t * G + g) * BLOCK_BYTES;
  *reinterpret_cast<uint4 *>(blk + lane * 16) = make_uint4(words[0], words[1], words[2], words[3]);
  if (tq == 0) {
    const int n0 = TILE_N * t + gq, n1 = n0 + 8;
    const uint32_t s0 = n0 < N ? sc[(size_t)n0 * G + g] : 0u;
    const uint32_t s1 = n1 < N ? sc[(size_t)n1 * G + g] : 0u;
    const uint32_t b0 = n0 < N ? bi[(size_t)n0 * G + g] : 0u;
    const uint32_t b1 = n1 < N ? bi[(size_t)n1 * G + g] : 0u;
    *reinterpret_cast<uint2 *>(blk + CODE_BYTES + gq * 8) =
        make_uint2(s0 | (s1 << 16), b0 | (b1 << 16));
  }
}

// ------------------------------------------------------------- kernel ---
struct Smem {
  uint64_t *full, *empty;
  uint8_t *ring, *xf;
  float *xs;
};

__device__ __forceinline__ Smem carve(uint8_t *base, int H) {
  Smem s;
  s.full = reinterpret_cast<uint64_t *>(base);
  s.empty = s.full + NSTAGE;
  s.ring = base + BAR_BYTES;
  s.xf = s.ring + NSTAGE * STAGE_BYTES;
  s.xs = reinterpret_cast<float *>(s.xf + MAX_SLICE_GROUPS * H * 1024);
  return s;
}

// Stage the activations of groups [gs0, gs0+ng) in MMA B-fragment order:
// xf[(g*H + h)*32 + lane][step s] = {x[m][16s+2tq..+1], x[m][16s+2tq+8..+9]}
// for m = 8h + gq, lane = 4gq + tq; rows m >= M are zero.  xs[g*16 + m] is
// the fp32 sum of the group's 64 activations (k order).
template <int H>
__device__ __forceinline__ void stage_x(const __nv_bfloat16 *__restrict__ x, int M, int K,
                                        int gs0, int ng, const Smem &sm, int tid) {
  const int items = 8 * H * ng;
  for (int it = tid; it < items; it += CWARPS * 32) {
    const int g = it % ng;
    const int m = it / ng;
    uint32_t v[32];
    if (m < M) {
      const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)m * K + (size_t)(gs0 + g) * GROUP);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 t = src[i];
        v[4 * i] = t.x;
        v[4 * i + 1] = t.y;
        v[4 * i + 2] = t.z;
        v[4 * i + 3] = t.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] = 0u;
    }
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      sum += bf16lo(v[i]);
      sum += bf16hi(v[i]);
    }
    sm.xs[g * 16 + m] = sum;
    const int h = m >> 3, gq = m & 7;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
#pragma unroll
      for (int tq = 0; tq < 4; ++tq) {
        const int ln = 4 * gq + tq;
        *reinterpret_cast<uint2 *>(sm.xf + ((g * H + h) * 32 + ln) * 32 + s * 8) =
            make_uint2(v[8 * s + tq], v[8 * s + tq + 4]);
      }
    }
  }
}

template <int H>
__device__ __forceinline__ void store_tile(void *y, int y_f32, int M, int N, int t, int lane,
                                           const float (&v)[H][4]) {
  const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int h = 0; h < H; ++h) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = TILE_N * t + gq + ((j & 2) ? 8 : 0);
      const int m = 8 * h + 2 * tq + (j & 1);
      if (m < M && n < N) {
        if (y_f32)
          static_cast<float *>(y)[(size_t)m * N + n] = v[h][j];
        else
          static_cast<__nv_bfloat16 *>(y)[(size_t)m * N + n] = __float2bfloat16_rn(v[h][j]);
      }
    }
  }
}

template <int H>
__global__ void __launch_bounds__(THREADS, 1)
    qmm_kernel(const __nv_bfloat16 *__restrict__ x, const uint8_t *__restrict__ packed, void *y,
               int y_f32, int M, int N, int K, Plan plan, float *__restrict__ part,
               unsigned *__restrict__ counters, unsigned *err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const Smem sm = carve(smem_raw, H);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NT = plan.NT, G = plan.G;
  const long long u0 = (long long)blockIdx.x * plan.units / plan.ctas;
  const long long u1 = (long long)(blockIdx.x + 1) * plan.units / plan.ctas;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSTAGE; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == CWARPS) {
    // ------------------------------------------------------- producer --
    if (lane != 0) return;
    const uint64_t pol = l2_evict_first_policy();
    bool ok = true;
    uint32_t q = 0;
    for (long long u = u0; u < u1 && ok;) {
      const int s = (int)(u / NT);
      const long long bend = lmin(lmin(u1, u + CWARPS), (long long)(s + 1) * NT);
      const int nb = (int)(bend - u);
      const int gs0 = s * plan.GS;
      const int ng = imin(G, gs0 + plan.GS) - gs0;
      const int nkb = (ng + KB_GROUPS - 1) / KB_GROUPS;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int gfirst = gs0 + kb * KB_GROUPS;
        const int gcnt = imin(KB_GROUPS, ng - kb * KB_GROUPS);
        for (int w = 0; w < nb && ok; ++w) {
          const int t = (int)(u + w - (long long)s * NT);
          const int slot = q % NSTAGE;
          const uint32_t round = q / NSTAGE;
          ok = mbar_wait(&sm.empty[slot], (round & 1) ^ 1, err);
          if (!ok) break;
          const uint32_t bytes = (uint32_t)gcnt * BLOCK_BYTES;
          mbar_arrive_expect_tx(&sm.full[slot], bytes);
          tma_load_1d(sm.ring + (size_t)slot * STAGE_BYTES,
                      packed + ((size_t)t * G + gfirst) * BLOCK_BYTES, bytes, &sm.full[slot], pol);
          ++q;
        }
      }
      u = bend;
    }
    if (!ok) {
      // Drain: do not leave the CTA while copies may still land in its
      // shared memory.
      const uint32_t first = q > (uint32_t)NSTAGE ? q - NSTAGE : 0u;
      for (uint32_t qq = first; qq < q; ++qq)
        mbar_wait(&sm.full[qq % NSTAGE], (qq / NSTAGE) & 1, err);
    }
    return;
  }

  // ------------------------------------------------------- consumers --
  pdl_wait();  // activations, outputs and workspace follow the predecessor
  const int tid = threadIdx.x;
  const int gq = lane >> 2, tq = lane & 3;
  bool ok = true;
  uint32_t q = 0;
  int cur_slice = -1;
  for (long long u = u0; u < u1;) {
    const int s = (int)(u / NT);
    const long long bend = lmin(lmin(u1, u + CWARPS), (long long)(s + 1) * NT);
    const int nb = (int)(bend - u);
    const int gs0 = s * plan.GS;
    const int ng = imin(G, gs0 + plan.GS) - gs0;
    const int nkb = (ng + KB_GROUPS - 1) / KB_GROUPS;
    if (s != cur_slice) {
      named_barrier(1, CWARPS * 32);
      stage_x<H>(x, M, K, gs0, ng, sm, tid);
      named_barrier(1, CWARPS * 32);
      cur_slice = s;
    }
    if (warp < nb) {
      const int t = (int)(u + warp - (long long)s * NT);
      float yv[H][4];
#pragma unroll
      for (int h = 0; h < H; ++h)
#pragma unroll
        for (int j = 0; j < 4; ++j) yv[h][j] = 0.f;

      for (int kb = 0; kb < nkb; ++kb) {
        const uint32_t qq = q + (uint32_t)(kb * nb + warp);
        const int slot = qq % NSTAGE;
        if (ok) ok = mbar_wait(&sm.full[slot], (qq / NSTAGE) & 1, err);
        if (!ok) continue;
        const int gcnt = imin(KB_GROUPS, ng - kb * KB_GROUPS);
        const uint8_t *st = sm.ring + (size_t)slot * STAGE_BYTES;
        for (int gi = 0; gi < gcnt; ++gi) {
          const uint8_t *blk = st + gi * BLOCK_BYTES;
          const uint4 wv = *reinterpret_cast<const uint4 *>(blk + lane * 16);
          const uint2 sb = *reinterpret_cast<const uint2 *>(blk + CODE_BYTES + gq * 8);
          const int gl = kb * KB_GROUPS + gi;
          uint4 xa[H], xb[H];
#pragma unroll
          for (int h = 0; h < H; ++h) {
            const uint8_t *xp = sm.xf + ((gl * H + h) * 32 + lane) * 32;
            xa[h] = *reinterpret_cast<const uint4 *>(xp);
            xb[h] = *reinterpret_cast<const uint4 *>(xp + 16);
          }
          float acc[H][4];
#pragma unroll
          for (int h = 0; h < H; ++h)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[h][j] = 0.f;
          const uint32_t wsteps[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
          for (int st4 = 0; st4 < 4; ++st4) {
            const uint32_t w = wsteps[st4];
            const uint32_t a0 = (w & 0x000F000Fu) | 0x43004300u;
            const uint32_t a1 = ((w >> 4) & 0x000F000Fu) | 0x43004300u;
            const uint32_t a2 = ((w >> 8) & 0x000F000Fu) | 0x43004300u;
            const uint32_t a3 = ((w >> 12) & 0x000F000Fu) | 0x43004300u;
#pragma unroll
            for (int h = 0; h < H; ++h) {
              const uint4 &xv = (st4 < 2) ? xa[h] : xb[h];
              const uint32_t b0 = (st4 & 1) ? xv.z : xv.x;
              const uint32_t b1 = (st4 & 1) ? xv.w : xv.y;
              mma_bf16_16816(acc[h], a0, a1, a2, a3, b0, b1);
            }
          }
          const float s0 = bf16lo(sb.x), s1 = bf16hi(sb.x);
          const float c0 = fmaf(-128.f, s0, bf16lo(sb.y));
          const float c1 = fmaf(-128.f, s1, bf16hi(sb.y));
#pragma unroll
          for (int h = 0; h < H; ++h) {
            const float2 xsv = *reinterpret_cast<const float2 *>(sm.xs + gl * 16 + 8 * h + 2 * tq);
            yv[h][0] = fmaf(s0, acc[h][0], fmaf(c0, xsv.x, yv[h][0]));
            yv[h][1] = fmaf(s0, acc[h][1], fmaf(c0, xsv.y, yv[h][1]));
            yv[h][2] = fmaf(s1, acc[h][2], fmaf(c1, xsv.x, yv[h][2]));
            yv[h][3] = fmaf(s1, acc[h][3], fmaf(c1, xsv.y, yv[h][3]));
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[slot]);
      }

      if (ok) {
        if (plan.S == 1) {
          store_tile<H>(y, y_f32, M, N, t, lane, yv);
        } else {
          float *pp = part + (((size_t)s * NT + t) * 32 + lane) * 8;
#pragma unroll
          for (int h = 0; h < H; ++h)
            *reinterpret_cast<float4 *>(pp + 4 * h) = make_float4(yv[h][0], yv[h][1], yv[h][2], yv[h][3]);
          __threadfence();
          __syncwarp();
          unsigned prev = 0;
          if (lane == 0) prev = atomicAdd(&counters[t], 1u);
          prev = __shfl_sync(0xffffffffu, prev, 0);
          if (prev == (unsigned)(plan.S - 1)) {
            __threadfence();
            float tot[H][4];
#pragma unroll
            for (int h = 0; h < H; ++h)
#pragma unroll
              for (int j = 0; j < 4; ++j) tot[h][j] = 0.f;
            for (int ss = 0; ss < plan.S; ++ss) {
              const float *src = part + (((size_t)ss * NT + t) * 32 + lane) * 8;
#pragma unroll
              for (int h = 0; h < H; ++h) {
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(src + 4 * h));
                tot[h][0] += v.x;
                tot[h][1] += v.y;
                tot[h][2] += v.z;
                tot[h][3] += v.w;
              }
            }
            store_tile<H>(y, y_f32, M, N, t, lane, tot);
            if (lane == 0) counters[t] = 0u;  // ready for the next call
          }
        }
      }
    }
    q += (uint32_t)(nkb * nb);
    u = bend;
  }
}

}  // namespace qmm
}  // namespace sv

using namespace sv;

extern "C" {

size_t qmm_packed_bytes(int N, int K, int group) {
  if (N < 1 || K < qmm::GROUP || K % qmm::GROUP != 0 || group != qmm::GROUP) return 0;
  const size_t NT = ((size_t)N + qmm::TILE_N - 1) / qmm::TILE_N;
  return NT * (size_t)(K / qmm::GROUP) * qmm::BLOCK_BYTES;
}

sv_status qmm_prepack(const uint32_t *wq, const void *scales, const void *biases, int N, int K,
                      int group, void *packed_out, size_t packed_bytes, sv_stream_t stream) {
  if (!wq || !scales || !biases || !packed_out) return SV_ERR_INVALID_ARG;
  if (N < 1 || K < 1 || group < 1) return SV_ERR_INVALID_ARG;
  if (group != qmm::GROUP || K % qmm::GROUP != 0) return SV_ERR_UNSUPPORTED;
  const size_t need = qmm_packed_bytes(N, K, group);
  if (packed_bytes < need) return SV_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(packed_out) % 16 != 0) return SV_ERR_INVALID_ARG;
  const int NT = (N + qmm::TILE_N - 1) / qmm::TILE_N, G = K / qmm::GROUP;
  const long long threads = (long long)NT * G * 32;
  const int block = 256;
  const long long grid = (threads + block - 1) / block;
  if (grid > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
  cudaError_t e = launch(qmm::prepack_kernel, dim3((unsigned)grid), dim3(block), 0,
                         reinterpret_cast<cudaStream_t>(stream), wq,
                         static_cast<const uint16_t *>(scales), static_cast<const uint16_t *>(biases),
                         N, K, NT, G, static_cast<uint8_t *>(packed_out));
  return from_cuda(e);
}

size_t qmm_workspace_bytes(int M, int N, int K) {
  (void)M;
  if (N < 1 || K < qmm::GROUP || K % qmm::GROUP != 0) return 0;
  const int sms = device_sm_count();
  if (sms <= 0) return 0;
  return qmm::workspace_bytes(qmm::make_plan(N, K, sms));
}

sv_status qmm_small_m(const void *x_bf16, const void *packed_w, void *y, sv_dtype y_dtype, int M,
                      int N, int K, int group, void *workspace, size_t ws_bytes,
                      sv_stream_t stream) {
  if (!x_bf16 || !packed_w || !y) return SV_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || group < 1) return SV_ERR_INVALID_ARG;
  if (y_dtype != SV_BF16 && y_dtype != SV_F32) return SV_ERR_INVALID_ARG;
  if (M > 16 || group != qmm::GROUP || K % qmm::GROUP != 0) return SV_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(x_bf16) % 16 != 0 || reinterpret_cast<uintptr_t>(packed_w) % 16 != 0)
    return SV_ERR_INVALID_ARG;
  const int sms = device_sm_count();
  if (sms <= 0) return SV_ERR_CUDA;
  const qmm::Plan plan = qmm::make_plan(N, K, sms);
  const size_t need = qmm::workspace_bytes(plan);
  if (need > 0 && (!workspace || ws_bytes < need)) return SV_ERR_WORKSPACE;
  unsigned *err = device_error_word();
  if (!err) return SV_ERR_CUDA;
  unsigned *counters = static_cast<unsigned *>(workspace);
  float *part = nullptr;
  if (need > 0) {
    const size_t cbytes = ((size_t)plan.NT * 4 + 255) / 256 * 256;
    part = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + cbytes);
  }
  const int yf = (y_dtype == SV_F32) ? 1 : 0;
  const auto *xp = static_cast<const __nv_bfloat16 *>(x_bf16);
  const auto *wp = static_cast<const uint8_t *>(packed_w);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (M <= 8)
    e = launch(qmm::qmm_kernel<1>, dim3(plan.ctas), dim3(qmm::THREADS), qmm::smem_bytes(1), s, xp,
               wp, y, yf, M, N, K, plan, part, counters, err);
  else
    e = launch(qmm::qmm_kernel<2>, dim3(plan.ctas), dim3(qmm::THREADS), qmm::smem_bytes(2), s, xp,
               wp, y, yf, M, N, K, plan, part, counters, err);
  return from_cuda(e);
}

}  // extern "C"
