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
#include "tcgen05.cuh"

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
  int stall_first;       // test aid: arm the first KV copy without issuing it (waits run out)
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
  // (no early launch_dependents: the combine is let in as this kernel's CTAs
  // exit; its CTAs waiting beside this latency-bound kernel slowed it)

  if (warp == NCW) {
    // ------------------------------------------------------- producer --
    if (lane != 0) return;
    // The committed prefix (slots before L - M) does not depend on the
    // predecessor kernel: it streams in while the predecessor drains, and
    // the wait comes before the first block that holds draft slots.
    const long long first_dep = ((long long)P.L - P.M) / BLK;
    bool waited = false;
    const uint64_t pol = l2_evict_first_policy();
    bool ok = true;
    uint32_t q = 0;
    for (long long u = u0; u < u1 && ok; ++u) {
      const int h = (int)(u / pl.NB), b = (int)(u % pl.NB);
      if (!waited && b >= first_dep) {
        pdl_wait();
        waited = true;
      }
      for (int kv = 0; kv < 2 && ok; ++kv) {
        const int slot = q % NSLOT;
        ok = mbar_wait(&empty[slot], ((q / NSLOT) & 1) ^ 1, P.err);
        if (!ok) break;
        mbar_arrive_expect_tx(&full[slot], SLOT);
        if (!(P.stall_first && q == 0)) {
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(ring + slot * SLOT + c * BLK * 128, kv ? &mapV : &mapK, 64 * c, BLK * b, h,
                        &full[slot], pol);
        }
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

// ------------------------------------------------ tcgen05 variant --------
// The same split and partials as attn_kernel, with both products on the
// 5th-generation tensor cores and their fp32 accumulators in tensor memory:
//  * warp 9 streams K and V blocks with TMA (as above); warp 8 allocates TMEM
//    and one of its threads issues the MMAs and the TMA load of each head's
//    Q tile; warps 0-7 are the row warps: TMEM lane = query row, and warps w
//    and w+4 share the 32 rows of lane quarter w % 4, each taking half of a
//    block's 64 scores (and half of O's columns at the rare rescale and at
//    the segment's end), so the pair exchanges one maximum per block.
//  * S = Q K^T for a 64-slot block: A = Q (128 padded rows x D, K-major,
//    128-byte swizzle), B = the K block; D/16 MMAs of 128 x 64 x 16 into one
//    of two 64-column TMEM buffers.
//  * O += P V: A = P (bf16, 128 x 64, stored by the row threads into one of
//    two 32-column TMEM buffers, two probabilities per column), B = the V block
//    read MN-major; four MMAs of 128 x D x 16 into D TMEM columns that stay
//    resident for the whole head segment.  With P in tensor memory the ring
//    takes the shared memory beside Q: five 32 KB slots at D = 256.
//  * The running maximum is raised only when a block's maximum exceeds it by
//    more than 2^8 (otherwise P values up to 256 are accumulated against the
//    old maximum), so O in TMEM is rescaled rarely and the row threads wait
//    for the previous block's PV product only then; the final O / l is the
//    same quantity either way.
constexpr int TC_ROWS = 128;       // query rows per MMA tile (TMEM lanes)
constexpr int TC_ROW_WARPS = 8;    // two per TMEM lane quarter
constexpr int TC_THREADS = (TC_ROW_WARPS + 2) * 32;
constexpr float TC_RESCALE = 8.f;  // log2 of the largest unnormalised P

template <int D>
struct TcLayout {
  static constexpr int SLOT = BLK * D * 2;
  static constexpr int NS = D == 256 ? 5 : 8;  // ring slots: what shared memory holds beside Q
  static constexpr int RING = 2048;            // barriers and the pair exchange below
  static constexpr int QS = RING + NS * SLOT;
  static constexpr int END = QS + TC_ROWS * D * 2;
  // O (D columns), two S buffers (64 each), two P buffers (32 each)
  static constexpr uint32_t TMEM_COLS = 512u;
  static_assert(D + 2 * BLK + 2 * (BLK / 2) <= 512, "tensor memory");
};

static size_t tc_smem_bytes(int D) {
  const size_t need = 1024 + (D == 256 ? TcLayout<256>::END : TcLayout<128>::END);
  // at least 120 KB, so that one CTA (and one TMEM allocation) per SM
  return need < 120 * 1024 ? 120 * 1024 : need;
}

template <int D>
__global__ void __launch_bounds__(TC_THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                   const __grid_constant__ CUtensorMap mapQ, const Params P) {
  using LY = TcLayout<D>;
  constexpr int SLOT = LY::SLOT;
  constexpr int NKS = D / 16;
  constexpr int HALF = BLK / 2;  // scores per row thread and block
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  constexpr int NS = LY::NS;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem);
  uint64_t *empty = full + NS;
  uint64_t *s_full = empty + NS;     // [2] per S buffer
  uint64_t *s_free = s_full + 2;     // [2]
  uint64_t *p_full = s_free + 2;     // [2] per P buffer
  uint64_t *o_done = p_full + 2;     // [2] PV of a block that used P buffer b done
  uint64_t *o_free = o_done + 2;     // row threads have read O (segment end)
  uint64_t *q_full = o_free + 1;     // Q of the segment's head landed (TMA)
  uint64_t *q_zero = q_full + 1;     // padding rows of the Q tile zeroed
  uint64_t *idle = q_zero + 1;       // every MMA issued so far has completed
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(idle + 1);
  float *xchg = reinterpret_cast<float *>(smem + 1024);  // [2 halves][128 rows]
  uint8_t *ring = smem + LY::RING;
  uint8_t *qs = smem + LY::QS;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Plan &pl = P.plan;
  const long long u0 = (long long)blockIdx.x * pl.units / pl.ctas;
  const long long u1 = (long long)(blockIdx.x + 1) * pl.units / pl.ctas;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], TC_ROW_WARPS);
      mbar_init(&p_full[i], TC_ROW_WARPS);
      mbar_init(&o_done[i], 1);
    }
    mbar_init(o_free, TC_ROW_WARPS);
    mbar_init(q_full, 1);
    mbar_init(q_zero, TC_ROW_WARPS);
    mbar_init(idle, 1);
    fence_barrier_init();
  }
  if (warp == TC_ROW_WARPS) {
    tc::tmem_alloc(tmem_slot, LY::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tmem_slot;
  const uint32_t tO = tbase, tS = tbase + D;  // S buffers at columns D and D + 64
  const uint32_t tP = tbase + D + 2 * BLK;     // P buffers at columns D + 128 and D + 160
  // (no early launch_dependents: the combine is let in once every CTA has
  // issued its last products, below; its CTAs waiting beside this kernel slowed it)

  if (warp == TC_ROW_WARPS + 1) {
    // ------------------------------------------------------- producer --
    if (lane != 0) return;
    // the committed prefix streams in before the predecessor completes (as
    // in attn_kernel)
    const long long first_dep = ((long long)P.L - P.M) / BLK;
    bool waited = false;
    const uint64_t pol = l2_evict_first_policy();
    bool ok = true;
    uint32_t q = 0;
    for (long long u = u0; u < u1 && ok; ++u) {
      const int h = (int)(u / pl.NB), b = (int)(u % pl.NB);
      if (!waited && b >= first_dep) {
        pdl_wait();
        waited = true;
      }
      for (int kv = 0; kv < 2 && ok; ++kv) {
        const int slot = q % NS;
        ok = mbar_wait(&empty[slot], ((q / NS) & 1) ^ 1, P.err);
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
      const uint32_t first = q > (uint32_t)NS ? q - NS : 0u;
      for (uint32_t qq = first; qq < q; ++qq) mbar_wait(&full[qq % NS], (qq / NS) & 1, P.err);
    }
    return;
  }

  if (warp == TC_ROW_WARPS) {
    // ---------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t IDS = tc::idesc_bf16_f32(TC_ROWS, BLK, false);
      constexpr uint32_t IDO = tc::idesc_bf16_f32(TC_ROWS, D, true);
      const uint32_t qs_a = smem_u32(qs), ring_a = smem_u32(ring);
      bool ok = true;
      uint32_t j = 0;  // block index over the CTA's whole range
      int seg = 0;
      auto issue_s = [&](uint32_t jj) {
        const uint32_t qk = 2 * jj, slot = qk % NS, sb = jj & 1, use = jj >> 1;
        if (ok) ok = spin_wait(&full[slot], (qk / NS) & 1, P.err);
        if (ok && use >= 1) ok = spin_wait(&s_free[sb], (use - 1) & 1, P.err);
        if (!ok) return;
        tc::fence_after_sync();
        const uint32_t kb = ring_a + slot * SLOT;
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
          const uint32_t off = (ks & 3) * 32;  // k16 step within a 128-byte row
          const uint64_t a = tc::smem_desc_sw128(qs_a + (ks >> 2) * TC_ROWS * 128 + off, 16, 1024);
          const uint64_t b = tc::smem_desc_sw128(kb + (ks >> 2) * BLK * 128 + off, 16, 1024);
          tc::mma_bf16(tS + sb * BLK, a, b, IDS, ks > 0);
        }
        tc::commit(&s_full[sb]);
        tc::commit(&empty[slot]);
      };
      pdl_wait();
      const uint64_t pol = l2_evict_first_policy();
      for (long long u = u0; u < u1 && ok; ++seg) {
        const int h = (int)(u / pl.NB);
        const long long useg_end = lmin(u1, (long long)(h + 1) * pl.NB);
        const uint32_t nb = (uint32_t)(useg_end - u);
        // Q tile of head h: rows i*G + jh by TMA, once the previous head's
        // products have completed
        if (seg > 0) {
          tc::commit(idle);
          ok = spin_wait(idle, (seg - 1) & 1, P.err);
          if (!ok) break;
        }
        mbar_arrive_expect_tx(q_full, (uint32_t)(P.R * D * 2));
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(qs + c * TC_ROWS * 128, &mapQ, 64 * c, h * P.G, 0, q_full, pol);
        if (seg == 0) ok = spin_wait(q_zero, 0, P.err);
        if (ok) ok = spin_wait(q_full, seg & 1, P.err);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t j0 = j;
        issue_s(j);
        for (uint32_t t = 0; t < nb && ok; ++t, ++j) {
          if (t + 1 < nb) issue_s(j + 1);
          const uint32_t qv = 2 * j + 1, slot = qv % NS, pb = j & 1;
          if (ok) ok = spin_wait(&full[slot], (qv / NS) & 1, P.err);
          if (ok) ok = spin_wait(&p_full[pb], (j >> 1) & 1, P.err);
          // O of the previous head read out before this head overwrites it
          if (ok && t == 0 && seg > 0) ok = spin_wait(o_free, (seg - 1) & 1, P.err);
          if (!ok) break;
          tc::fence_after_sync();
          const uint32_t vb = ring_a + slot * SLOT;
#pragma unroll
          for (int ks = 0; ks < BLK / 16; ++ks) {
            const uint64_t b = tc::smem_desc_sw128(vb + ks * 2 * 1024, BLK * 128, 1024);
            tc::mma_bf16_ts(tO, tP + pb * (BLK / 2) + ks * 8, b, IDO, j > j0 || ks > 0);
          }
          tc::commit(&o_done[pb]);
          tc::commit(&empty[slot]);
        }
        u = useg_end;
      }
      // The combine may be scheduled once every CTA has issued its last
      // products: it waits for this grid to complete, and its small CTAs are
      // resident only for this kernel's tail (O read out, partials written).
      pdl_launch_dependents();
      // every MMA issued above has completed before TMEM is released
      tc::commit(idle);
      spin_wait(idle, (seg > 0 ? seg - 1 : 0) & 1, P.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ row warps (0-7) --
    pdl_wait();
    const int quarter = warp & 3, hf = warp >> 2;  // lane quarter, half of the columns
    const int r = quarter * 32 + lane;              // query row = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int L = P.L, M = P.M, G = P.G, R = P.R;
    const int RP = num_mtiles(R) * 16;
    const int vi = r / G;  // verify row of this query row
    const long long last = (long long)L - M + vi;
    const uint32_t dmask = (P.mask && vi < M) ? P.mask[vi] : 0u;
    const float sl2e = P.sl2e;
    const int pair_bar = 2 + quarter;  // named barrier of warps w and w+4
    // the Q tile's rows R..127 stay zero (TMA writes rows below R only)
    for (int idx = threadIdx.x; idx < (TC_ROWS - R) * (D / 8); idx += TC_ROW_WARPS * 32) {
      const int rr = R + idx / (D / 8), c = idx % (D / 8);
      *reinterpret_cast<uint4 *>(qs + swz(rr, c, TC_ROWS)) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) mbar_arrive(q_zero);
    bool ok = true;
    uint32_t j = 0;
    int seg = 0;
    for (long long u = u0; u < u1; ++seg) {
      const int h = (int)(u / pl.NB);
      const int b0 = (int)(u % pl.NB);
      const long long useg_end = lmin(u1, (long long)(h + 1) * pl.NB);
      const int b1 = (int)(useg_end - (long long)h * pl.NB);

      float m_use = -INFINITY, l_half = 0.f;
      const uint32_t j0 = j;
      for (int b = b0; b < b1; ++b, ++j) {
        // Every row warp runs every barrier of the loop whatever `ok` says
        // (the pair barriers have no time limit); after a timed-out wait
        // only the work is skipped.
        const uint32_t sb = j & 1;
        if (ok) ok = spin_wait(&s_full[sb], (j >> 1) & 1, P.err);
        ok = __all_sync(0xffffffffu, ok);
        tc::fence_after_sync();
        uint32_t raw[HALF];
        if (ok) {
          tc::ld32(tS + sb * BLK + hf * HALF + lane_off, raw);
          tc::wait_ld();
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[sb]);

        // ---- mask (blocks reaching the drafts or kv_len only), maximum ----
        const long long pos0 = (long long)BLK * b + hf * HALF;
        float s[HALF];
#pragma unroll
        for (int c = 0; c < HALF; ++c) s[c] = ok ? __uint_as_float(raw[c]) : 0.f;
        if ((long long)BLK * b + BLK - 1 > (long long)L - M) {
#pragma unroll
          for (int c = 0; c < HALF; ++c) {
            const long long pos = pos0 + c;
            bool hide;
            if (P.mask) {
              const long long t = pos - ((long long)L - M);
              hide = pos >= L || (t >= 0 && !((dmask >> t) & 1u));
            } else {
              hide = pos > last || pos >= L;
            }
            if (hide) s[c] = -INFINITY;
          }
        }
        float mx = s[0];
#pragma unroll
        for (int c = 1; c < HALF; ++c) mx = fmaxf(mx, s[c]);
        // the pair's maximum (raw scores; the scale is positive); the second
        // barrier keeps the slots until both have been read
        xchg[hf * TC_ROWS + r] = mx;
        named_barrier(pair_bar, 64);
        mx = fmaxf(mx, xchg[(hf ^ 1) * TC_ROWS + r]) * sl2e;
        named_barrier(pair_bar, 64);
        // raise the base only when the block's maximum is far above it
        float alpha = 1.f;
        if (mx > m_use + TC_RESCALE) {
          alpha = (m_use == -INFINITY) ? 0.f : exp2f(m_use - mx);
          m_use = mx;
        }
        const float nbase = (m_use == -INFINITY) ? 0.f : -m_use;

        // ---- P = exp2(S * scale - base) ----
        float sum = 0.f;
        uint32_t pk[HALF / 2];
#pragma unroll
        for (int e = 0; e < HALF / 2; ++e) {
          const float p0 = ex2_approx(fmaf(s[2 * e], sl2e, nbase));
          const float p1 = ex2_approx(fmaf(s[2 * e + 1], sl2e, nbase));
          sum += p0 + p1;
          pk[e] = pack_bf16x2(p0, p1);
        }
        l_half = alpha * l_half + sum;

        // P buffer j&1 free once the PV of block j-2 is done
        if (ok && j >= j0 + 2) ok = spin_wait(&o_done[j & 1], ((j - 2) >> 1) & 1, P.err);
        ok = __all_sync(0xffffffffu, ok);
        // rescale this warp's half of O after the PV of block j-1
        if (ok && j > j0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          ok = spin_wait(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1, P.err);
          ok = __all_sync(0xffffffffu, ok);
          tc::fence_after_sync();
          if (ok) {
#pragma unroll 1
            for (int c0 = hf * (D / 2); c0 < (hf + 1) * (D / 2); c0 += 32) {
              uint32_t o[32];
              tc::ld32(tO + c0 + lane_off, o);
              tc::wait_ld();
#pragma unroll
              for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
              tc::st32(tO + c0 + lane_off, o);
            }
            tc::wait_st();
          }
        }
        if (ok) {
          // this warp's half of the row: columns hf*16 .. hf*16+15 of P buffer j&1
          tc::st16(tP + (j & 1) * (BLK / 2) + hf * (HALF / 2) + lane_off, pk);
          tc::wait_st();
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[j & 1]);
      }

      // ---- segment partial: unnormalised O, base (log2) and sum ----
      if (ok && j >= j0 + 2) {
        ok = spin_wait(&o_done[(j - 2) & 1], ((j - 2) >> 1) & 1, P.err);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok && j > j0) {
        ok = spin_wait(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1, P.err);
        ok = __all_sync(0xffffffffu, ok);
      }
      tc::fence_after_sync();
      // the pair's sums
      xchg[hf * TC_ROWS + r] = l_half;
      named_barrier(pair_bar, 64);
      const float l_run = l_half + xchg[(hf ^ 1) * TC_ROWS + r];
      named_barrier(pair_bar, 64);
      if (ok) {
        const size_t slot = (size_t)blockIdx.x * pl.maxseg + seg;
        float *op = P.opart + (slot * RP + r) * D;
#pragma unroll 1
        for (int c0 = hf * (D / 2); c0 < (hf + 1) * (D / 2); c0 += 32) {
          uint32_t o[32];
          tc::ld32(tO + c0 + lane_off, o);
          tc::wait_ld();
          if (r < R) {
#pragma unroll
            for (int c = 0; c < 32; c += 4)
              *reinterpret_cast<uint4 *>(op + c0 + c) = make_uint4(o[c], o[c + 1], o[c + 2], o[c + 3]);
          }
        }
        if (r < R && hf == 0) {
          float *mlp = P.ml + (slot * RP + r) * 2;
          mlp[0] = m_use;
          mlp[1] = l_run;
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
      u = useg_end;
    }
  }
  // row warps and the MMA issuer meet here; warp 8 then releases TMEM
  tc::fence_before_sync();
  named_barrier(1, (TC_ROW_WARPS + 1) * 32);
  if (warp == TC_ROW_WARPS) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tbase, LY::TMEM_COLS);
  }
}

// Merge the head-segment partials of every (query row, KV head) and write O.
// One block per (row, head, 128 columns of D) (more blocks in flight for what
// is a latency-bound gather).  Each thread finds its own segment's slot and
// (max, sum) directly; the weights exp2(m_s - max) and the denominator use
// fixed shuffle trees; warp w adds the weighted partial rows of segments
// w, w+8, ... and the eight warp sums are added in warp order.  Every order is
// fixed, so the result is deterministic.  The partial rows of the first
// COMBINE_CH * 8 segments are loaded together with the (max, sum) pairs,
// before the weights are known, so the block waits for memory once.
constexpr int COMBINE_THREADS = 256;
constexpr int COMBINE_WARPS = COMBINE_THREADS / 32;
constexpr int COMBINE_MAXSEG = 256;
constexpr int COMBINE_COLS = 128;  // columns of D per block (a warp's 32 lanes x 4)
constexpr int COMBINE_CH = 8;      // segments in flight per lane

__global__ void __launch_bounds__(COMBINE_THREADS) combine_kernel(const Params P) {
  __shared__ float s_w[COMBINE_MAXSEG];
  __shared__ float s_red[COMBINE_WARPS], s_den[COMBINE_WARPS];
  __shared__ __align__(16) float s_part[COMBINE_WARPS][COMBINE_COLS];
  pdl_launch_dependents();
  pdl_wait();
  const int r = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
  const int c0 = blockIdx.z * COMBINE_COLS;  // first column of D this block adds
  const int warp = tid >> 5, lane = tid & 31;
  const int D = P.D, RP = num_mtiles(P.R) * 16;
  const Plan &pl = P.plan;
  // CTAs whose unit ranges meet head h: the owners of its first and last
  // unit (CTA c owns units [c*units/ctas, (c+1)*units/ctas)); 32-bit
  // divisions when the products fit, since they precede every load
  const bool narrow = (long long)pl.units * pl.ctas < (1LL << 31);
  const long long ulo = (long long)h * pl.NB, uhi = ulo + pl.NB - 1;
  auto owner = [&](long long u) {
    return narrow ? (int)(((unsigned)(u + 1) * (unsigned)pl.ctas - 1u) / (unsigned)pl.units)
                  : (int)(((u + 1) * pl.ctas - 1) / pl.units);
  };
  const int c_first = owner(ulo), c_last = owner(uhi);
  const int n = imin(c_last - c_first + 1, COMBINE_MAXSEG);
  // Partial slot of segment si: CTA c_first + si, its segment for head h.
  // Every CTA after c_first starts inside head h (its first unit lies in
  // (ulo, uhi]), so only c_first's segment index can be above zero.
  const int cu0 = narrow ? (int)((unsigned)c_first * (unsigned)pl.units / (unsigned)pl.ctas)
                         : (int)((long long)c_first * pl.units / pl.ctas);
  const int seg0 = h - cu0 / pl.NB;
  auto slot_of = [&](int si) { return (c_first + si) * pl.maxseg + (si == 0 ? seg0 : 0); };
  auto load_row = [&](int si) {
    return __ldcg(reinterpret_cast<const float4 *>(P.opart + ((size_t)slot_of(si) * RP + r) * D + c0 +
                                                   (size_t)lane * 4));
  };
  float4 v[COMBINE_CH];
#pragma unroll
  for (int i = 0; i < COMBINE_CH; ++i) {
    const int si = warp + i * COMBINE_WARPS;
    v[i] = si < n ? load_row(si) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float m = -INFINITY, l = 0.f;
  if (tid < n) {
    const int slot = slot_of(tid);
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
  // warp sums over its segments: lane holds 4 consecutive columns
  float acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = 0.f;
  for (int s0 = warp; s0 < n; s0 += COMBINE_CH * COMBINE_WARPS) {
    float wv[COMBINE_CH];
    if (s0 != warp) {  // rounds after the first: load now
#pragma unroll
      for (int i = 0; i < COMBINE_CH; ++i) {
        const int si = s0 + i * COMBINE_WARPS;
        v[i] = si < n ? load_row(si) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int i = 0; i < COMBINE_CH; ++i) {
      const int si = s0 + i * COMBINE_WARPS;
      wv[i] = si < n ? s_w[si] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < COMBINE_CH; ++i) {
      acc[0] = fmaf(wv[i], v[i].x, acc[0]);
      acc[1] = fmaf(wv[i], v[i].y, acc[1]);
      acc[2] = fmaf(wv[i], v[i].z, acc[2]);
      acc[3] = fmaf(wv[i], v[i].w, acc[3]);
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) s_part[warp][lane * 4 + k] = acc[k];
  __syncthreads();
  const float inv = 1.f / den;
  const int i = r / P.G, j = r % P.G;
  for (int d = tid; d < COMBINE_COLS; d += COMBINE_THREADS) {
    float num = s_part[0][d];
#pragma unroll
    for (int w = 1; w < COMBINE_WARPS; ++w) num += s_part[w][d];
    P.o[((size_t)i * P.Hq + (size_t)h * P.G + j) * D + c0 + d] = __float2bfloat16_rn(num * inv);
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

// 3-D map over the queries [M][Hq][D] bf16: dims (D, Hq, M), box (64, G, M),
// 128-byte swizzle; one box per 64 columns is the G*M rows of one KV head.
bool make_q_map(CUtensorMap *map, const void *q, int D, int Hq, int M, int G) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)M};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Hq * D * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)M};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_tc(const CUtensorMap &mk, const CUtensorMap &mv, const Params &P, cudaStream_t s) {
  CUtensorMap mq;
  if (!make_q_map(&mq, P.q, D, P.Hq, P.M, P.G)) return cudaErrorInvalidValue;
  return launch(attn_tc_kernel<D>, dim3(P.plan.ctas), dim3(TC_THREADS), tc_smem_bytes(D), s, mk, mv, mq,
                P);
}

// Query rows per KV head from which the tcgen05 kernel is the default: up to
// one m16 tile the mma.sync kernel's shorter per-block chain streams the
// cache faster; from two tiles its warp-level MMAs and per-tile softmax
// exchanges cost about as much as or more than the tensor-memory pipeline,
// whose time hardly depends on the number of rows.
constexpr int TC_MIN_ROWS = 17;

static bool use_tc(int R) {
  const unsigned f = launch_flags();
  if (f & SV_LAUNCH_ATTN_MMA_SYNC) return false;
  if (f & SV_LAUNCH_ATTN_TCGEN05) return true;
  return R >= TC_MIN_ROWS;
}

static cudaError_t launch_any(int D, int MT, const CUtensorMap &mk, const CUtensorMap &mv,
                              const Params &P, cudaStream_t s) {
  if (use_tc(P.R)) return D == 256 ? launch_tc<256>(mk, mv, P, s) : launch_tc<128>(mk, mv, P, s);
  return D == 256 ? launch_mt<256>(MT, mk, mv, P, s) : launch_mt<128>(MT, mk, mv, P, s);
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
  P.stall_first = (launch_flags() & SV_LAUNCH_TEST_STALL_COPY) ? 1 : 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  e = attn::launch_any(D, MT, mk, mv, P, s);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  e = launch(attn::combine_kernel, dim3(R, Hkv, D / attn::COMBINE_COLS), dim3(attn::COMBINE_THREADS), 0,
             s, P);
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
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SV_ERR_CUDA;
  void *scratch = noalloc_scratch(dev);
  if (!scratch) return SV_ERR_CUDA;
  // the same checks and launches as verify_attn, with the fixed array as the
  // workspace: a shape whose partials exceed it is refused (SV_ERR_WORKSPACE)
  // before anything is launched
  return verify_attn_run(q, k_cache, v_cache, o, M, Hq, Hkv, D, kv_len, kv_stride_tokens, scale,
                         nullptr, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
