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
constexpr int BAR_BYTES = 1024;
constexpr int QUAD = 4;            // groups in flight per warp (independent MMA chains)

// Activation rows of one K slice live in shared memory: 8*H rows (H = 1 for
// M <= 8, 2 for M <= 16) of up to 80/H groups, so the slice length depends on
// H only.  Rows are padded by 16 bytes (row stride = 16 mod 128) so that the
// per-lane 16-byte fragment loads are free of bank conflicts.
__host__ __device__ constexpr int max_slice_groups(int H) { return 80 / H; }
__host__ __device__ constexpr int xrow_stride(int H) { return max_slice_groups(H) * 128 + 16; }

struct Plan {
  int NT;     // 16-row tiles
  int G;      // groups per row
  int S;      // K slices
  int GS;     // groups per slice (the last may be shorter)
  int units;  // S * NT (slice-major)
  int ctas;   // grid size
};

// Split plan for an N x K matrix read by 8*H-row activation blocks on `sms`
// SMs: the number of K slices minimises the bytes streamed by the busiest SM
// (plus one block's worth per split partial).  Depends on N, K, H and the SM
// count only, so every M in 1..8 (and every M in 9..16) runs the same plan.
static Plan make_plan(int N, int K, int H, int sms) {
  Plan p{};
  p.NT = (N + TILE_N - 1) / TILE_N;
  p.G = K / GROUP;
  const int msg = max_slice_groups(H);
  const int smin = (p.G + msg - 1) / msg;
  double best = 1e300;
  for (int S = smin; S <= p.G && S <= 64; ++S) {
    const int GS = (p.G + S - 1) / S;
    const int Se = (p.G + GS - 1) / GS;
    if (Se != S) continue;  // every slice non-empty
    const long long units = (long long)S * p.NT;
    const int ctas = (int)std::min<long long>(units, sms);
    const long long per = (units + ctas - 1) / ctas;
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
  return BAR_BYTES + (size_t)NSTAGE * STAGE_BYTES + (size_t)8 * H * xrow_stride(H) +
         (size_t)max_slice_groups(H) * 16 * sizeof(float) + 1024;
}

static size_t workspace_bytes(const Plan &p) {
  if (p.S <= 1) return 0;
  const size_t counters = ((size_t)p.NT * 4 + 255) / 256 * 256;
  return counters + (size_t)p.S * p.NT * 32 * 8 * sizeof(float);
}

// ----------------------------------------------------------- prepack ---
// One thread per (tile, group, lane).  For k16 step s of the group, lane
// (gq = lane/4, tq = lane%4) holds one word whose nibble j is the code of
//   row gq + 8*(j&1),  k = 16*tq + 4*s + 2*((j>>1)&1) + ((j>>2)&1)
// so that (w >> 4i) & 0x000F000F is MMA A-fragment register i.  The MMA's
// logical k order is thereby permuted within the group so that the B fragment
// of step s is the four activations x[16tq+4s .. 16tq+4s+3]: each lane's B
// fragments for the whole group are 32 contiguous bytes of the activation row.
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
      const int kk = 16 * tq + 4 * s + ((j & 2) ? 2 : 0) + ((j & 4) ? 1 : 0);
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
  uint64_t *full, *empty, *xfull, *xempty;
  uint8_t *ring, *xraw;
  float *xs;
};

__device__ __forceinline__ Smem carve(uint8_t *base, int H) {
  Smem s;
  s.full = reinterpret_cast<uint64_t *>(base);
  s.empty = s.full + NSTAGE;
  s.xfull = s.empty + NSTAGE;
  s.xempty = s.xfull + 1;
  s.ring = base + BAR_BYTES;
  s.xraw = s.ring + NSTAGE * STAGE_BYTES;
  s.xs = reinterpret_cast<float *>(s.xraw + 8 * H * xrow_stride(H));
  return s;
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

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Batch bookkeeping shared by producer and consumers: units [u, bend) of one
// slice s, one unit per consumer warp.
struct Batch {
  int s, nb, gs0, ng, nkb;
  long long bend;
};
__device__ __forceinline__ Batch batch_at(long long u, long long u1, const Plan &pl) {
  Batch b;
  b.s = (int)(u / pl.NT);
  b.bend = lmin(lmin(u1, u + CWARPS), (long long)(b.s + 1) * pl.NT);
  b.nb = (int)(b.bend - u);
  b.gs0 = b.s * pl.GS;
  b.ng = imin(pl.G, b.gs0 + pl.GS) - b.gs0;
  b.nkb = (b.ng + KB_GROUPS - 1) / KB_GROUPS;
  return b;
}

template <int H>
__global__ void __launch_bounds__(THREADS, 1)
    qmm_kernel(const __nv_bfloat16 *__restrict__ x, const uint8_t *__restrict__ packed, void *y,
               int y_f32, int M, int N, int K, Plan plan, float *__restrict__ part,
               unsigned *__restrict__ counters, unsigned *err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const Smem sm = carve(base, H);
  constexpr int XS = xrow_stride(H);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NT = plan.NT, G = plan.G;
  const long long u0 = (long long)blockIdx.x * plan.units / plan.ctas;
  const long long u1 = (long long)(blockIdx.x + 1) * plan.units / plan.ctas;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSTAGE; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], 1);
    }
    mbar_init(sm.xfull, 1);
    mbar_init(sm.xempty, CWARPS);
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
    int x_issued = 0;       // activation slices loaded so far
    int x_want = -1;        // slice whose activations are still to be loaded
    bool waited = false;    // predecessor grid awaited (activations are its output)
    int last_slice = -1;    // slice of the previous batch
    auto issue_x = [&](int slice) {
      const int gs0 = slice * plan.GS;
      const int ng = imin(G, gs0 + plan.GS) - gs0;
      mbar_arrive_expect_tx(sm.xfull, (uint32_t)(M * ng * 128));
      for (int m = 0; m < M; ++m)
        tma_load_1d(sm.xraw + (size_t)m * XS, x + (size_t)m * K + (size_t)gs0 * GROUP,
                    (uint32_t)(ng * 128), sm.xfull, pol);
      ++x_issued;
      x_want = -1;
    };
    // Load slice `x_want` once the consumers have released the previous one.
    auto poll_x = [&](bool block) -> bool {
      if (x_want < 0) return true;
      if (x_issued == 0) {
        if (!waited) {
          pdl_wait();
          waited = true;
        }
        issue_x(x_want);
        return true;
      }
      const uint32_t par = (uint32_t)(x_issued - 1) & 1u;
      if (mbar_try_wait(sm.xempty, par) || (block && mbar_wait(sm.xempty, par, err))) {
        issue_x(x_want);
        return true;
      }
      return !block;
    };
    for (long long u = u0; u < u1 && ok;) {
      const Batch b = batch_at(u, u1, plan);
      if (b.s != last_slice) {
        // a new slice: finish any pending activation load first
        if (x_want >= 0) ok = poll_x(true);
        x_want = b.s;
        last_slice = b.s;
      }
      for (int kb = 0; kb < b.nkb && ok; ++kb) {
        const int gfirst = b.gs0 + kb * KB_GROUPS;
        const int gcnt = imin(KB_GROUPS, b.ng - kb * KB_GROUPS);
        for (int w = 0; w < b.nb && ok; ++w) {
          const int t = (int)(u + w - (long long)b.s * NT);
          const int slot = q % NSTAGE;
          const uint32_t par = ((q / NSTAGE) & 1) ^ 1;
          if (q == NSTAGE && x_issued == 0) poll_x(true);  // first ring fill done
          // wait for the slot, loading pending activations meanwhile
          if (!mbar_try_wait(&sm.empty[slot], par)) {
            const long long t0 = clock64();
            while (!mbar_try_wait(&sm.empty[slot], par)) {
              if (x_issued > 0) poll_x(false);
              if (clock64() - t0 > WAIT_LIMIT_CYCLES) {
                atomicOr(err, ERR_TIMEOUT);
                ok = false;
                break;
              }
            }
            if (!ok) break;
          }
          if (x_issued > 0) poll_x(false);
          const uint32_t bytes = (uint32_t)gcnt * BLOCK_BYTES;
          mbar_arrive_expect_tx(&sm.full[slot], bytes);
          tma_load_1d(sm.ring + (size_t)slot * STAGE_BYTES,
                      packed + ((size_t)t * G + gfirst) * BLOCK_BYTES, bytes, &sm.full[slot], pol);
          ++q;
        }
      }
      u = b.bend;
    }
    if (ok) ok = poll_x(true);
    if (!ok) {
      // Drain: do not leave while copies may still land in shared memory.
      const uint32_t first = q > (uint32_t)NSTAGE ? q - NSTAGE : 0u;
      for (uint32_t qq = first; qq < q; ++qq)
        mbar_wait(&sm.full[qq % NSTAGE], (qq / NSTAGE) & 1, err);
      if (x_issued > 0) mbar_wait(sm.xfull, (uint32_t)(x_issued - 1) & 1u, err);
    }
    return;
  }

  // ------------------------------------------------------- consumers --
  pdl_wait();  // outputs and workspace follow the predecessor
  const int tid = threadIdx.x;
  const int gq = lane >> 2, tq = lane & 3;
  // rows M..8H-1 of the activation buffer are never loaded: zero them once
  for (int i = tid; i < (8 * H - M) * (XS / 16); i += CWARPS * 32) {
    const int r = M + i / (XS / 16), c = i % (XS / 16);
    *reinterpret_cast<uint4 *>(sm.xraw + (size_t)r * XS + c * 16) = make_uint4(0u, 0u, 0u, 0u);
  }
  bool ok = true;
  uint32_t q = 0;
  int cur_slice = -1, xk = 0;
  for (long long u = u0; u < u1;) {
    const Batch b = batch_at(u, u1, plan);
    if (b.s != cur_slice) {
      if (cur_slice >= 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.xempty);  // done with the old activations
      }
      if (ok) ok = mbar_wait(sm.xfull, (uint32_t)xk & 1u, err);
      ++xk;
      named_barrier(1, CWARPS * 32);  // old group sums no longer read
      // per-group activation sums (fp32, k order)
      for (int it = tid; it < 8 * H * b.ng; it += CWARPS * 32) {
        const int m = it / b.ng, g = it % b.ng;
        const uint8_t *row = sm.xraw + (size_t)m * XS + (size_t)g * 128;
        float sum = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 v = *reinterpret_cast<const uint4 *>(row + 16 * i);
          sum += bf16lo(v.x);
          sum += bf16hi(v.x);
          sum += bf16lo(v.y);
          sum += bf16hi(v.y);
          sum += bf16lo(v.z);
          sum += bf16hi(v.z);
          sum += bf16lo(v.w);
          sum += bf16hi(v.w);
        }
        sm.xs[g * 16 + m] = sum;
      }
      named_barrier(1, CWARPS * 32);
      cur_slice = b.s;
    }
    if (warp < b.nb) {
      const int t = (int)(u + warp - (long long)b.s * NT);
      float yv[H][4];
#pragma unroll
      for (int h = 0; h < H; ++h)
#pragma unroll
        for (int j = 0; j < 4; ++j) yv[h][j] = 0.f;
      const uint8_t *xlane = sm.xraw + (size_t)gq * XS + 32 * tq;

      for (int kb = 0; kb < b.nkb; ++kb) {
        const uint32_t qq = q + (uint32_t)(kb * b.nb + warp);
        const int slot = qq % NSTAGE;
        if (ok) ok = mbar_wait(&sm.full[slot], (qq / NSTAGE) & 1, err);
        if (!ok) continue;
        const int gcnt = imin(KB_GROUPS, b.ng - kb * KB_GROUPS);
        const uint8_t *st = sm.ring + (size_t)slot * STAGE_BYTES;
        for (int g0 = 0; g0 < gcnt; g0 += QUAD) {
          const int cnt = imin(QUAD, gcnt - g0);
          uint4 wv[QUAD];
          uint2 sb[QUAD];
          uint4 xa[QUAD][H], xb[QUAD][H];
          float acc[QUAD][H][4];
#pragma unroll
          for (int qd = 0; qd < QUAD; ++qd) {
            if (qd < cnt) {
              const uint8_t *blk = st + (g0 + qd) * BLOCK_BYTES;
              wv[qd] = *reinterpret_cast<const uint4 *>(blk + lane * 16);
              sb[qd] = *reinterpret_cast<const uint2 *>(blk + CODE_BYTES + gq * 8);
              const int gl = kb * KB_GROUPS + g0 + qd;
#pragma unroll
              for (int h = 0; h < H; ++h) {
                const uint8_t *xp = xlane + (size_t)(8 * h) * XS + (size_t)gl * 128;
                xa[qd][h] = *reinterpret_cast<const uint4 *>(xp);
                xb[qd][h] = *reinterpret_cast<const uint4 *>(xp + 16);
              }
            }
#pragma unroll
            for (int h = 0; h < H; ++h)
#pragma unroll
              for (int j = 0; j < 4; ++j) acc[qd][h][j] = 0.f;
          }
#pragma unroll
          for (int st4 = 0; st4 < 4; ++st4) {
#pragma unroll
            for (int qd = 0; qd < QUAD; ++qd) {
              if (qd < cnt) {
                const uint32_t w = st4 == 0 ? wv[qd].x : st4 == 1 ? wv[qd].y : st4 == 2 ? wv[qd].z : wv[qd].w;
                const uint32_t a0 = (w & 0x000F000Fu) | 0x43004300u;
                const uint32_t a1 = ((w >> 4) & 0x000F000Fu) | 0x43004300u;
                const uint32_t a2 = ((w >> 8) & 0x000F000Fu) | 0x43004300u;
                const uint32_t a3 = ((w >> 12) & 0x000F000Fu) | 0x43004300u;
#pragma unroll
                for (int h = 0; h < H; ++h) {
                  const uint4 &xv = (st4 < 2) ? xa[qd][h] : xb[qd][h];
                  const uint32_t b0 = (st4 & 1) ? xv.z : xv.x;
                  const uint32_t b1 = (st4 & 1) ? xv.w : xv.y;
                  mma_bf16_16816(acc[qd][h], a0, a1, a2, a3, b0, b1);
                }
              }
            }
          }
#pragma unroll
          for (int qd = 0; qd < QUAD; ++qd) {
            if (qd < cnt) {
              const int gl = kb * KB_GROUPS + g0 + qd;
              const float s0 = bf16lo(sb[qd].x), s1 = bf16hi(sb[qd].x);
              const float c0 = fmaf(-128.f, s0, bf16lo(sb[qd].y));
              const float c1 = fmaf(-128.f, s1, bf16hi(sb[qd].y));
#pragma unroll
              for (int h = 0; h < H; ++h) {
                const float2 xsv = *reinterpret_cast<const float2 *>(sm.xs + gl * 16 + 8 * h + 2 * tq);
                yv[h][0] = fmaf(s0, acc[qd][h][0], fmaf(c0, xsv.x, yv[h][0]));
                yv[h][1] = fmaf(s0, acc[qd][h][1], fmaf(c0, xsv.y, yv[h][1]));
                yv[h][2] = fmaf(s1, acc[qd][h][2], fmaf(c1, xsv.x, yv[h][2]));
                yv[h][3] = fmaf(s1, acc[qd][h][3], fmaf(c1, xsv.y, yv[h][3]));
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[slot]);
      }

      if (ok) {
        if (plan.S == 1) {
          store_tile<H>(y, y_f32, M, N, t, lane, yv);
        } else {
          float *pp = part + (((size_t)b.s * NT + t) * 32 + lane) * 8;
#pragma unroll
          for (int h = 0; h < H; ++h)
            *reinterpret_cast<float4 *>(pp + 4 * h) = make_float4(yv[h][0], yv[h][1], yv[h][2], yv[h][3]);
          fence_acq_rel_gpu();  // release this lane's partial
          __syncwarp();
          unsigned prev = 0;
          if (lane == 0) prev = atomicAdd(&counters[t], 1u);
          prev = __shfl_sync(0xffffffffu, prev, 0);
          if (prev == (unsigned)(plan.S - 1)) {
            fence_acq_rel_gpu();  // acquire the other slices' partials
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
    q += (uint32_t)(b.nkb * b.nb);
    u = b.bend;
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
  const int H = M > 8 ? 2 : 1;
  return qmm::workspace_bytes(qmm::make_plan(N, K, H, sms));
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
  const int H = M > 8 ? 2 : 1;
  const qmm::Plan plan = qmm::make_plan(N, K, H, sms);
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
