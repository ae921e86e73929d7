// attn.cu -- multi-row verify attention over a bf16 GQA KV cache.
//
// For verify row i (0..M-1) and query head h:
//   O[i][h] = softmax_j(scale * <Q[i][h], K[g][j]>) V[g][j],  j <= L-M+i,
//   g = h / (Hq/Hkv).
// All M rows and all Hq/Hkv query heads of a KV head are scored against each
// KV tile while it sits in shared memory, so the cache is read from HBM once
// per verify pass ("Speculative decoding and MTP on Apple silicon", Facts:
// Metal's decode attention re-reads the KV cache once per query row; the
// multi-row kernel reads each KV tile once; flash-decoding verify kernel).
//
// Design (GB300):
//  * Flash-decoding split: the (KV head, 64-slot block) units are divided
//    evenly over one CTA per SM; each CTA keeps a running (max, sum, O) per
//    query row for each head segment it covers and writes it as a partial;
//    a small combine kernel merges the partials per (row, head).
//  * A producer warp streams K and V blocks with TMA tensor copies
//    (128-byte swizzle, zero fill past kv_len) into a 4-slot ring.
//  * The R = M*Hq/Hkv query rows form MT = ceil(R/16) m16 tiles; each tile is
//    owned by a group of four warps.  A warp keeps its Q fragments in
//    registers, computes S for 16 of the 64 slots (m16n8k16 bf16 MMA, fp32),
//    the group exchanges row maxima and sums through shared memory, writes P
//    as bf16, and each warp then accumulates O for a quarter of D.
//  * Scores are kept in the log2 domain (scale * log2 e folded in); the
//    causal mask among the drafts is applied only to blocks that reach past
//    slot L-M.
#include <mutex>

#include "common.cuh"

namespace sv {
namespace attn {

constexpr int BLK = 64;    // KV slots per block
constexpr int NSLOT = 4;   // ring slots (each one K or one V block)
constexpr int MAX_MT = 6;  // up to 96 query rows per KV head (M = 16 at 6 heads per group)

struct Plan {
  int NB;      // blocks per head
  int units;   // Hkv * NB
  int ctas;
  int maxseg;  // head segments per CTA
};

static Plan make_plan(int Hkv, long long L, int sms) {
  Plan p{};
  p.NB = (int)((L + BLK - 1) / BLK);
  p.units = Hkv * p.NB;
  p.ctas = imin(p.units, sms);
  const int per = (p.units + p.ctas - 1) / p.ctas;
  p.maxseg = imin(Hkv, (per + p.NB - 1) / p.NB + 1);
  return p;
}

__host__ __device__ inline int num_mtiles(int R) { return (R + 15) / 16; }

static size_t smem_bytes(int D, int MT) {
  const size_t slot = (size_t)BLK * D * 2;
  return 2048 + NSLOT * slot + (size_t)MT * 16 * D * 2 + 2 * (size_t)MT * 2048 +
         2 * 2 * (size_t)MT * 4 * 16 * sizeof(float);
}

static size_t workspace_bytes(const Plan &p, int MT, int D) {
  const size_t slots = (size_t)p.ctas * p.maxseg;
  return slots * (size_t)MT * 16 * ((size_t)D + 2) * sizeof(float);
}

struct Params {
  const __nv_bfloat16 *q;
  __nv_bfloat16 *o;
  float *opart;  // [slots][R_pad][D]
  float *ml;     // [slots][R_pad][2]
  unsigned *err;
  int M, Hq, Hkv, G, R, D;
  int L;
  float sl2e;  // scale * log2(e)
  Plan plan;
  const uint32_t *mask;  // draft tree [M] (bit j: draft slot L-M+j visible); null: the chain
};

// Byte offset of 16-byte chunk `c` (of D/8) in row `r` of a tile stored as
// D/64 swizzled boxes of [rows][128 B] (TMA SWIZZLE_128B layout).
__device__ __forceinline__ uint32_t swz(int r, int c, int rows) {
  return (uint32_t)((c >> 3) * rows * 128 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

template <int D, int MT>
__global__ void __launch_bounds__((4 * MT + 1) * 32, 1)
    attn_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                const Params P) {
  constexpr int NCW = 4 * MT;  // consumer warps
  constexpr int SLOT = BLK * D * 2;
  constexpr int RP = MT * 16;  // padded query rows
  constexpr int NKS = D / 16;  // k16 steps over D
  constexpr int NTW = D / 32;  // n8 tiles of O per warp (a quarter of D)
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 128-byte-swizzled TMA tiles need a 1024-byte aligned base
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *empty = full + NSLOT;
  uint8_t *ring = smem + 1024;
  uint8_t *qs = ring + NSLOT * SLOT;
  uint8_t *ps = qs + RP * D * 2;
  float *red_max = reinterpret_cast<float *>(ps + 2 * MT * 2048);  // [2][MT][4][16]
  float *red_sum = red_max + 2 * MT * 64;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Plan &pl = P.plan;
  const long long u0 = (long long)blockIdx.x * pl.units / pl.ctas;
  const long long u1 = (long long)(blockIdx.x + 1) * pl.units / pl.ctas;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], NCW);
    }
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();

  if (warp == NCW) {
    // ------------------------------------------------------- producer --
    if (lane != 0) return;
    pdl_wait();
    const uint64_t pol = l2_evict_first_policy();
    bool ok = true;
    uint32_t q = 0;
    for (long long u = u0; u < u1 && ok; ++u) {
      const int h = (int)(u / pl.NB), b = (int)(u % pl.NB);
      for (int kv = 0; kv < 2 && ok; ++kv) {
        const int slot = q % NSLOT;
        ok = mbar_wait(&empty[slot], ((q / NSLOT) & 1) ^ 1, P.err);
        if (!ok) break;
        mbar_arrive_expect_tx(&full[slot], SLOT);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(ring + slot * SLOT + c * BLK * 128, kv ? &mapV : &mapK, 64 * c, BLK * b, h,
                      &full[slot], pol);
        ++q;
      }
    }
    if (!ok) {
      const uint32_t first = q > (uint32_t)NSLOT ? q - NSLOT : 0u;
      for (uint32_t qq = first; qq < q; ++qq) mbar_wait(&full[qq % NSLOT], (qq / NSLOT) & 1, P.err);
    }
    return;
  }

  // --------------------------------------------------------- consumers --
  pdl_wait();
  const int g = warp >> 2;   // m-tile (query rows 16g..16g+15)
  const int jw = warp & 3;   // slots 16jw..16jw+15 of a block; quarter jw of D
  const int gq = lane >> 2, tq = lane & 3;
  const int ctid = threadIdx.x;  // consumers are threads 0..NCW*32-1
  const int L = P.L, M = P.M, G = P.G, R = P.R;
  const int row0 = 16 * g + gq, row1 = row0 + 8;
  const int i0 = row0 / G, i1 = row1 / G;  // verify row of each query row
  const long long last0 = (long long)L - M + i0, last1 = (long long)L - M + i1;
  // draft-tree masks of this lane's two query rows (padding rows see no draft)
  const uint32_t mask0 = (P.mask && i0 < M) ? P.mask[i0] : 0u;
  const uint32_t mask1 = (P.mask && i1 < M) ? P.mask[i1] : 0u;
  uint8_t *pbase = ps + g * 2048;
  float *rmax = red_max + g * 64, *rsum = red_sum + g * 64;
  const int dchunk0 = jw * (D / 32);  // first 8-column chunk of this warp's quarter of D

  bool ok = true;
  uint32_t q = 0;
  int buf = 0;
  int seg_j = 0;
  for (long long u = u0; u < u1; ++seg_j) {
    const int h = (int)(u / pl.NB);
    const int b0 = (int)(u % pl.NB);
    const long long useg_end = lmin(u1, (long long)(h + 1) * pl.NB);
    const int b1 = (int)(useg_end - (long long)h * pl.NB);

    // ---- stage Q for KV head h (rows r = i*G + j, j < G) ----
    named_barrier(1, NCW * 32);
    for (int idx = ctid; idx < RP * (D / 8); idx += NCW * 32) {
      const int r = idx / (D / 8), c = idx % (D / 8);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (r < R) {
        const int i = r / G, j = r % G;
        v = *reinterpret_cast<const uint4 *>(P.q + ((size_t)i * P.Hq + (size_t)h * G + j) * D + c * 8);
      }
      *reinterpret_cast<uint4 *>(qs + swz(r, c, RP)) = v;
    }
    named_barrier(1, NCW * 32);
    // Q fragments: kept in registers, or (three or more m-tiles: 12 to 24
    // consumer warps, 128 to 72 registers a thread) re-read from shared
    // memory at each k16 step
    constexpr bool QREG = MT < 3;
    constexpr int NQR = QREG ? NKS : 1;
    uint32_t qa[NQR][4];
    const int qr = 16 * g + (lane & 7) + 8 * ((lane >> 3) & 1);
    if (QREG) {
#pragma unroll
      for (int ks = 0; ks < NQR; ++ks) {
        const int c = 2 * ks + (lane >> 4);
        ldmatrix_x4(qa[ks], smem_u32(qs + swz(qr, c, RP)));
      }
    }

    float m_run0 = -INFINITY, m_run1 = -INFINITY, l_run0 = 0.f, l_run1 = 0.f;
    float oacc[NTW][4];
#pragma unroll
    for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) oacc[nt][j] = 0.f;

    for (int b = b0; b < b1; ++b) {
      // ------------------------------------------- S = Q K^T (16 slots) --
      const int slotK = q % NSLOT;
      if (ok) ok = mbar_wait(&full[slotK], (q / NSLOT) & 1, P.err);
      float sacc[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) sacc[nt][j] = 0.f;
      if (ok) {
        const uint8_t *kslot = ring + slotK * SLOT;
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
          const int pos = 16 * jw + 8 * (lane >> 4) + (lane & 7);
          const int c = 2 * ks + ((lane >> 3) & 1);
          uint32_t kb[4];
          ldmatrix_x4(kb, smem_u32(kslot + swz(pos, c, BLK)));
          uint32_t qf[4];
          if (QREG) {
#pragma unroll
            for (int t = 0; t < 4; ++t) qf[t] = qa[QREG ? ks : 0][t];
          } else {
            ldmatrix_x4(qf, smem_u32(qs + swz(qr, 2 * ks + (lane >> 4), RP)));
          }
          mma_bf16_16816(sacc[0], qf[0], qf[1], qf[2], qf[3], kb[0], kb[1]);
          mma_bf16_16816(sacc[1], qf[0], qf[1], qf[2], qf[3], kb[2], kb[3]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slotK]);
      }
      ++q;

      // ------------------------------------------- mask, block row max --
      const long long pbase_pos = (long long)BLK * b + 16 * jw + 2 * tq;
      const bool need_mask = (long long)BLK * b + BLK - 1 > (long long)L - M;
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const long long pos = pbase_pos + 8 * nt + (j & 1);
          float v = sacc[nt][j] * P.sl2e;
          if (need_mask) {
            bool hide;
            if (P.mask) {
              const long long t = pos - ((long long)L - M);  // draft slot index, < M <= 32
              hide = pos >= L || (t >= 0 && !((((j & 2) ? mask1 : mask0) >> t) & 1u));
            } else {
              const long long last = (j & 2) ? last1 : last0;
              hide = pos > last || pos >= L;
            }
            if (hide) v = -INFINITY;
          }
          sacc[nt][j] = v;
        }
        mx0 = fmaxf(mx0, fmaxf(sacc[nt][0], sacc[nt][1]));
        mx1 = fmaxf(mx1, fmaxf(sacc[nt][2], sacc[nt][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      float *rm = rmax + buf * MT * 64;
      float *rs = rsum + buf * MT * 64;
      if (tq == 0) {
        rm[jw * 16 + gq] = mx0;
        rm[jw * 16 + gq + 8] = mx1;
      }
      named_barrier(2 + g, 128);
      float bm0 = rm[gq], bm1 = rm[gq + 8];
#pragma unroll
      for (int w = 1; w < 4; ++w) {
        bm0 = fmaxf(bm0, rm[w * 16 + gq]);
        bm1 = fmaxf(bm1, rm[w * 16 + gq + 8]);
      }
      const float mn0 = fmaxf(m_run0, bm0), mn1 = fmaxf(m_run1, bm1);
      const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
      const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
      const float alpha0 = exp2f(m_run0 - base0), alpha1 = exp2f(m_run1 - base1);

      // ------------------------------------------- P = exp2(S - m), sums --
      float sum0 = 0.f, sum1 = 0.f;
      uint8_t *pb = pbase + buf * MT * 2048;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const float p0 = exp2f(sacc[nt][0] - base0), p1 = exp2f(sacc[nt][1] - base0);
        const float p2 = exp2f(sacc[nt][2] - base1), p3 = exp2f(sacc[nt][3] - base1);
        sum0 += p0 + p1;
        sum1 += p2 + p3;
        const int chunk = 2 * jw + nt;
        *reinterpret_cast<uint32_t *>(pb + gq * 128 + ((chunk ^ (gq & 7)) << 4) + 4 * tq) =
            pack_bf16x2(p0, p1);
        *reinterpret_cast<uint32_t *>(pb + (gq + 8) * 128 + ((chunk ^ (gq & 7)) << 4) + 4 * tq) =
            pack_bf16x2(p2, p3);
      }
      sum0 += __shfl_xor_sync(0xffffffffu, sum0, 1);
      sum0 += __shfl_xor_sync(0xffffffffu, sum0, 2);
      sum1 += __shfl_xor_sync(0xffffffffu, sum1, 1);
      sum1 += __shfl_xor_sync(0xffffffffu, sum1, 2);
      if (tq == 0) {
        rs[jw * 16 + gq] = sum0;
        rs[jw * 16 + gq + 8] = sum1;
      }
      named_barrier(2 + g, 128);
      float bs0 = 0.f, bs1 = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        bs0 += rs[w * 16 + gq];
        bs1 += rs[w * 16 + gq + 8];
      }
      l_run0 = alpha0 * l_run0 + bs0;
      l_run1 = alpha1 * l_run1 + bs1;
      m_run0 = mn0;
      m_run1 = mn1;

      // ------------------------------------------- O += P V (quarter of D) --
      const int slotV = q % NSLOT;
      if (ok) ok = mbar_wait(&full[slotV], (q / NSLOT) & 1, P.err);
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) {
        oacc[nt][0] *= alpha0;
        oacc[nt][1] *= alpha0;
        oacc[nt][2] *= alpha1;
        oacc[nt][3] *= alpha1;
      }
      if (ok) {
        const uint8_t *vslot = ring + slotV * SLOT;
#pragma unroll
        for (int ks = 0; ks < BLK / 16; ++ks) {
          uint32_t pa[4];
          {
            const int r = (lane & 7) + 8 * ((lane >> 3) & 1);
            const int c = 2 * ks + (lane >> 4);
            ldmatrix_x4(pa, smem_u32(pb + r * 128 + (((c) ^ (r & 7)) << 4)));
          }
#pragma unroll
          for (int ntp = 0; ntp < NTW / 2; ++ntp) {
            const int pos = 16 * ks + 8 * ((lane >> 3) & 1) + (lane & 7);
            const int c = dchunk0 + 2 * ntp + (lane >> 4);
            uint32_t vb[4];
            ldmatrix_x4_trans(vb, smem_u32(vslot + swz(pos, c, BLK)));
            mma_bf16_16816(oacc[2 * ntp], pa[0], pa[1], pa[2], pa[3], vb[0], vb[1]);
            mma_bf16_16816(oacc[2 * ntp + 1], pa[0], pa[1], pa[2], pa[3], vb[2], vb[3]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slotV]);
      }
      ++q;
      buf ^= 1;
    }

    // ---- segment partial: unnormalised O, running max (log2) and sum ----
    if (ok) {
      const size_t slot = (size_t)blockIdx.x * pl.maxseg + seg_j;
      float *op = P.opart + slot * RP * D;
#pragma unroll
      for (int nt = 0; nt < NTW; ++nt) {
        const int d = 8 * (dchunk0 + nt) + 2 * tq;
        *reinterpret_cast<float2 *>(op + (size_t)row0 * D + d) = make_float2(oacc[nt][0], oacc[nt][1]);
        *reinterpret_cast<float2 *>(op + (size_t)row1 * D + d) = make_float2(oacc[nt][2], oacc[nt][3]);
      }
      if (jw == 0 && tq == 0) {
        float *mlp = P.ml + slot * RP * 2;
        mlp[row0 * 2] = m_run0;
        mlp[row0 * 2 + 1] = l_run0;
        mlp[row1 * 2] = m_run1;
        mlp[row1 * 2 + 1] = l_run1;
      }
    }
    u = useg_end;
  }
}

// Merge the head-segment partials of every (query row, KV head) and write O.
// One block per (row, head).  Each thread finds its own segment's slot and
// (max, sum) directly; the weights exp2(m_s - max) and the denominator use
// fixed shuffle trees; warp w adds the weighted partial rows of segments
// w, w+8, ... with all of its loads in flight, and the eight warp sums are
// added in warp order.  Every order is fixed, so the result is deterministic.
constexpr int COMBINE_THREADS = 256;
constexpr int COMBINE_WARPS = COMBINE_THREADS / 32;
constexpr int COMBINE_MAXSEG = 256;

__global__ void __launch_bounds__(COMBINE_THREADS) combine_kernel(const Params P) {
  __shared__ int s_slot[COMBINE_MAXSEG];
  __shared__ float s_w[COMBINE_MAXSEG];
  __shared__ float s_red[COMBINE_WARPS], s_den[COMBINE_WARPS];
  __shared__ __align__(16) float s_part[COMBINE_WARPS][256];
  pdl_launch_dependents();
  pdl_wait();
  const int r = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int D = P.D, RP = num_mtiles(P.R) * 16;
  const Plan &pl = P.plan;
  // CTAs whose unit ranges meet head h: the owners of its first and last unit
  const long long ulo = (long long)h * pl.NB, uhi = ulo + pl.NB - 1;
  const int c_first = (int)(((ulo + 1) * pl.ctas - 1) / pl.units);
  const int c_last = (int)(((uhi + 1) * pl.ctas - 1) / pl.units);
  const int n = imin(c_last - c_first + 1, COMBINE_MAXSEG);
  float m = -INFINITY, l = 0.f;
  if (tid < n) {
    const int cc = c_first + tid;
    const long long cu0 = (long long)cc * pl.units / pl.ctas;
    const int slot = cc * pl.maxseg + (h - (int)(cu0 / pl.NB));
    s_slot[tid] = slot;
    m = P.ml[((size_t)slot * RP + r) * 2];
    l = P.ml[((size_t)slot * RP + r) * 2 + 1];
  }
  float mx = m;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if (lane == 0) s_red[warp] = mx;
  __syncthreads();
  float mstar = s_red[0];
#pragma unroll
  for (int w = 1; w < COMBINE_WARPS; ++w) mstar = fmaxf(mstar, s_red[w]);
  const float wgt = (tid < n && m != -INFINITY) ? exp2f(m - mstar) : 0.f;
  if (tid < n) s_w[tid] = wgt;
  float wl = wgt * l;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wl += __shfl_xor_sync(0xffffffffu, wl, off);
  if (lane == 0) s_den[warp] = wl;
  __syncthreads();
  float den = s_den[0];
#pragma unroll
  for (int w = 1; w < COMBINE_WARPS; ++w) den += s_den[w];
  // warp sums over its segments: lane holds D/32 consecutive columns
  const int cpl = D / 32;  // 4 or 8
  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = 0.f;
  constexpr int CH = 4;  // segments in flight per lane
  for (int s0 = warp; s0 < n; s0 += CH * COMBINE_WARPS) {
    float4 v[CH][2];
    float wv[CH];
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      const int si = s0 + i * COMBINE_WARPS;
      wv[i] = 0.f;
      v[i][0] = v[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (si < n) {
        wv[i] = s_w[si];
        const float4 *src = reinterpret_cast<const float4 *>(
            P.opart + ((size_t)s_slot[si] * RP + r) * D + (size_t)lane * cpl);
        v[i][0] = __ldcg(src);
        if (cpl == 8) v[i][1] = __ldcg(src + 1);
      }
    }
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      acc[0] = fmaf(wv[i], v[i][0].x, acc[0]);
      acc[1] = fmaf(wv[i], v[i][0].y, acc[1]);
      acc[2] = fmaf(wv[i], v[i][0].z, acc[2]);
      acc[3] = fmaf(wv[i], v[i][0].w, acc[3]);
      acc[4] = fmaf(wv[i], v[i][1].x, acc[4]);
      acc[5] = fmaf(wv[i], v[i][1].y, acc[5]);
      acc[6] = fmaf(wv[i], v[i][1].z, acc[6]);
      acc[7] = fmaf(wv[i], v[i][1].w, acc[7]);
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k)
    if (k < cpl) s_part[warp][lane * cpl + k] = acc[k];
  __syncthreads();
  const float inv = 1.f / den;
  const int i = r / P.G, j = r % P.G;
  for (int d = tid; d < D; d += COMBINE_THREADS) {
    float num = s_part[0][d];
#pragma unroll
    for (int w = 1; w < COMBINE_WARPS; ++w) num += s_part[w][d];
    P.o[((size_t)i * P.Hq + (size_t)h * P.G + j) * D + d] = __float2bfloat16_rn(num * inv);
  }
}

// ------------------------------------------------------------ host side --
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) ==
            cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D map over a [Hkv][stride][D] bf16 cache: dims (D, L, Hkv), box
// (64, 64, 1), 128-byte swizzle, zero fill beyond L.
bool make_kv_map(CUtensorMap *map, const void *base, int D, long long L, long long stride, int Hkv) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)Hkv};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)stride * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)BLK, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, int MT>
cudaError_t launch_attn(const CUtensorMap &mk, const CUtensorMap &mv, const Params &P, cudaStream_t s) {
  return launch(attn_kernel<D, MT>, dim3(P.plan.ctas), dim3((4 * MT + 1) * 32), smem_bytes(D, MT), s,
                mk, mv, P);
}

// The kernel for MT query m-tiles (1 <= MT <= MAX_MT).
template <int D>
cudaError_t launch_mt(int MT, const CUtensorMap &mk, const CUtensorMap &mv, const Params &P,
                      cudaStream_t s) {
  switch (MT) {
    case 1: return launch_attn<D, 1>(mk, mv, P, s);
    case 2: return launch_attn<D, 2>(mk, mv, P, s);
    case 3: return launch_attn<D, 3>(mk, mv, P, s);
    case 4: return launch_attn<D, 4>(mk, mv, P, s);
    case 5: return launch_attn<D, 5>(mk, mv, P, s);
    case 6: return launch_attn<D, 6>(mk, mv, P, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace attn
}  // namespace sv

using namespace sv;

extern "C" {

size_t verify_attn_workspace_bytes(int M, int Hq, int Hkv, int D, int64_t kv_len) {
  if (M < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || kv_len < M) return 0;
  const int sms = device_sm_count();
  if (sms <= 0) return 0;
  const int R = M * (Hq / Hkv);
  const attn::Plan p = attn::make_plan(Hkv, kv_len, sms);
  return attn::workspace_bytes(p, attn::num_mtiles(R), D);
}

}  // extern "C"

// verify_attn and verify_attn_masked (mask null: the chain of drafts).
static sv_status verify_attn_run(const void *q, const void *k_cache, const void *v_cache, void *o,
                                 int M, int Hq, int Hkv, int D, int64_t kv_len,
                                 int64_t kv_stride_tokens, float scale, const uint32_t *mask,
                                 void *workspace, size_t ws_bytes, sv_stream_t stream) {
  if (!q || !k_cache || !v_cache || !o) return SV_ERR_INVALID_ARG;
  if (M < 1 || Hq < 1 || Hkv < 1 || D < 1 || Hq % Hkv != 0) return SV_ERR_INVALID_ARG;
  if (kv_len < M || kv_stride_tokens < kv_len) return SV_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY)) return SV_ERR_INVALID_ARG;
  if (D != 128 && D != 256) return SV_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  const int R = M * G;
  if (R > 16 * attn::MAX_MT) return SV_ERR_UNSUPPORTED;
  if (kv_len > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
  for (const void *p : {q, k_cache, v_cache, (const void *)o})
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return SV_ERR_INVALID_ARG;
  const int sms = device_sm_count();
  if (sms <= 0) return SV_ERR_CUDA;
  const attn::Plan plan = attn::make_plan(Hkv, kv_len, sms);
  const int MT = attn::num_mtiles(R);
  const size_t need = attn::workspace_bytes(plan, MT, D);
  if (!workspace || ws_bytes < need) return SV_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return SV_ERR_INVALID_ARG;
  CUtensorMap mk, mv;
  if (!attn::make_kv_map(&mk, k_cache, D, kv_len, kv_stride_tokens, Hkv) ||
      !attn::make_kv_map(&mv, v_cache, D, kv_len, kv_stride_tokens, Hkv))
    return SV_ERR_CUDA;
  attn::Params P{};
  P.q = static_cast<const __nv_bfloat16 *>(q);
  P.o = static_cast<__nv_bfloat16 *>(o);
  P.opart = static_cast<float *>(workspace);
  P.ml = P.opart + (size_t)plan.ctas * plan.maxseg * MT * 16 * D;
  P.err = device_error_word();
  if (!P.err) return SV_ERR_CUDA;
  P.M = M;
  P.Hq = Hq;
  P.Hkv = Hkv;
  P.G = G;
  P.R = R;
  P.D = D;
  P.L = (int)kv_len;
  P.sl2e = scale * 1.4426950408889634f;
  P.plan = plan;
  P.mask = mask;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  e = D == 256 ? attn::launch_mt<256>(MT, mk, mv, P, s) : attn::launch_mt<128>(MT, mk, mv, P, s);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  e = launch(attn::combine_kernel, dim3(R, Hkv), dim3(attn::COMBINE_THREADS), 0, s, P);
  return from_cuda(e);
}

extern "C" {

sv_status verify_attn(const void *q, const void *k_cache, const void *v_cache, void *o, int M, int Hq,
                      int Hkv, int D, int64_t kv_len, int64_t kv_stride_tokens, float scale,
                      void *workspace, size_t ws_bytes, sv_stream_t stream) {
  return verify_attn_run(q, k_cache, v_cache, o, M, Hq, Hkv, D, kv_len, kv_stride_tokens, scale,
                         nullptr, workspace, ws_bytes, stream);
}

sv_status verify_attn_masked(const void *q, const void *k_cache, const void *v_cache, void *o, int M,
                             int Hq, int Hkv, int D, int64_t kv_len, int64_t kv_stride_tokens,
                             float scale, const uint32_t *draft_mask, void *workspace,
                             size_t ws_bytes, sv_stream_t stream) {
  if (!draft_mask || reinterpret_cast<uintptr_t>(draft_mask) % 4 != 0) return SV_ERR_INVALID_ARG;
  if (M > 32) return SV_ERR_UNSUPPORTED;
  return verify_attn_run(q, k_cache, v_cache, o, M, Hq, Hkv, D, kv_len, kv_stride_tokens, scale,
                         draft_mask, workspace, ws_bytes, stream);
}

}  // extern "C"

// ------------------------------------------------ allocation-free variant --
// Some callers cannot allocate device memory when they need to run the
// attention: a plugin called from inside another engine's enqueue, code that
// runs between a capture's begin and end where cudaMalloc is not allowed, or a
// service that fixes its device-memory budget at start-up.  For them the
// split-KV partials of verify_attn live in this fixed array instead of a
// caller-supplied workspace.  Every GPU that loads the library holds it (16
// MiB) until the process exits.
namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64] = {};

// Device address of the array on the current device, looked up once per
// device with that device current (host code cannot use the symbol itself).
void *noalloc_scratch(int dev) {
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" {

sv_status verify_attn_noalloc(const void *q, const void *k_cache, const void *v_cache, void *o,
                              int M, int Hq, int Hkv, int D, int64_t kv_len,
                              int64_t kv_stride_tokens, float scale, sv_stream_t stream) {
  if (!q || !k_cache || !v_cache || !o) return SV_ERR_INVALID_ARG;
  if (M < 1 || Hq < 1 || Hkv < 1 || D < 1 || Hq % Hkv != 0) return SV_ERR_INVALID_ARG;
  if (kv_len < M || kv_stride_tokens < kv_len) return SV_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY)) return SV_ERR_INVALID_ARG;
  if (D != 128 && D != 256) return SV_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  const int R = M * G;
  if (R > 16 * attn::MAX_MT) return SV_ERR_UNSUPPORTED;
  if (kv_len > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
  for (const void *p : {q, k_cache, v_cache, (const void *)o})
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return SV_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SV_ERR_CUDA;
  const int sms = device_sm_count();
  if (sms <= 0) return SV_ERR_CUDA;
  const attn::Plan plan = attn::make_plan(Hkv, kv_len, sms);
  const int MT = attn::num_mtiles(R);
  if (attn::workspace_bytes(plan, MT, D) > kNoAllocScratchBytes) return SV_ERR_WORKSPACE;
  void *scratch = noalloc_scratch(dev);
  if (!scratch) return SV_ERR_CUDA;
  CUtensorMap mk, mv;
  if (!attn::make_kv_map(&mk, k_cache, D, kv_len, kv_stride_tokens, Hkv) ||
      !attn::make_kv_map(&mv, v_cache, D, kv_len, kv_stride_tokens, Hkv))
    return SV_ERR_CUDA;
  attn::Params P{};
  P.q = static_cast<const __nv_bfloat16 *>(q);
  P.o = static_cast<__nv_bfloat16 *>(o);
  P.opart = static_cast<float *>(scratch);
  P.ml = P.opart + (size_t)plan.ctas * plan.maxseg * MT * 16 * D;
  P.err = device_error_word();
  if (!P.err) return SV_ERR_CUDA;
  P.M = M;
  P.Hq = Hq;
  P.Hkv = Hkv;
  P.G = G;
  P.R = R;
  P.D = D;
  P.L = (int)kv_len;
  P.sl2e = scale * 1.4426950408889634f;
  P.plan = plan;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  e = D == 256 ? attn::launch_mt<256>(MT, mk, mv, P, s) : attn::launch_mt<128>(MT, mk, mv, P, s);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  e = launch(attn::combine_kernel, dim3(R, Hkv), dim3(attn::COMBINE_THREADS), 0, s, P);
  return from_cuda(e);
}

}  // extern "C"
