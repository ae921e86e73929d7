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
//  * Prepacked layout: 16-row tiles are grouped in batches of 8; for every
//    group of 64 k the batch's 8 tiles sit side by side (a 4.5 KB
//    "group-block"), then the next group.  Each tile's 576 bytes hold the
//    codes arranged as MMA A fragments (512 B) and the 16 rows' scales and
//    biases (64 B).  A CTA therefore reads one contiguous byte range, which
//    keeps the DRAM access stream sequential.
//  * One CTA per SM: a producer warp streams the CTA's range of group-blocks
//    with TMA bulk copies (16 group-blocks = 72 KB per stage, a ring as deep
//    as shared memory allows: two stages at M <= 8) from the CTA's start --
//    the weights do not depend on the predecessor kernel -- and sixteen
//    consumer warps, four per pair of tiles, each take every fourth group of
//    a stage.  At the end of a batch segment the four warps' sums are added
//    in shared memory.  How the matrix is divided over the CTAs:
//      - whole batches per CTA when there are at least as many batches as
//        SMs: nothing is merged across CTAs;
//      - a thread-block cluster per batch when its clusters fit: the
//        cluster's CTAs split the batch's groups and add their sums through
//        distributed shared memory, in rank order;
//      - a batch split over a few CTAs whose ranges stay inside it, merged by
//        the batch's last CTA to arrive, which adds the partials in CTA order;
//      - otherwise the even stream-K split, where a batch cut by CTA
//        boundaries is merged the same way.  An arrival warp makes the
//        arrival for a range's cut first batch mid-range, so the consumers'
//        range ends with at most one arrival.
//    Every order is fixed, so results are deterministic.
//  * Dequantisation is one LOP3 per pair of codes: (code | 0x6400) is the
//    fp16 value 1024 + code, exact, and (code << 4 | 0x6400) is 1024 +
//    16 code, so the four A registers of a k16 step come from one word with
//    one shift (8-bit codes: a whole byte per fp16 register, one MMA per
//    step).  The MMA (m16n8k16, fp16 -> fp32) computes sum_k x*(1024+f q) per
//    group on activations converted to fp16 (times 2^-6, once per window);
//    the affine terms are folded per group:
//       sum_k x*(s*q + b) = (64 s / f) * acc + (b - 1024 s / f) * sum_k x,
//    with 64 s / f stored by the prepack (a power-of-two scaling, exact).
//  * The activation rows of the CTA's K window are loaded by TMA into shared
//    memory (the first window by a consumer thread as soon as the predecessor
//    kernel has completed); the prepack permutes k within each group so that a lane's B
//    fragments for a group are 32 contiguous bytes of a row, shared by both
//    of the warp's tiles.  M <= 8 uses one n8 half of the MMA, M <= 16 two;
//    lanes of padding rows read a row of zeros.
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>

#include "common.cuh"

namespace sv {
namespace qmm {

constexpr int TILE_N = 16;
constexpr int GROUP = 64;
constexpr int BLOCK_BYTES = 576;     // one tile x one group: 512 B codes + 64 B scales/biases
constexpr int CODE_BYTES = 512;
constexpr int BATCH = 8;             // tiles per batch
constexpr int TPW = 2;               // tiles per consumer warp
constexpr int PAIRS = BATCH / TPW;   // tile pairs per batch
constexpr int CWARPS = 16;           // consumer warps
constexpr int GSPLIT = CWARPS / PAIRS;  // warps per tile pair, splitting the groups
constexpr int THREADS = (CWARPS + 2) * 32;  // + the producer warp and the arrival warp
constexpr int GB_BYTES = BATCH * BLOCK_BYTES;  // one group-block (4608 B)
// Byte layout of one tile x one group and of a group-block for 4-bit and
// 8-bit codes (8-bit: two 512-byte halves of codes, then the 64 bytes of
// scales and biases).
template <int BITS>
struct Pack {
  static constexpr int CODE = BITS == 8 ? 2 * CODE_BYTES : CODE_BYTES;
  static constexpr int BLOCK = CODE + 64;
  static constexpr int GB = BATCH * BLOCK;
};

// Activations enter the MMAs as fp16 scaled by 2^-6 (exact for bf16 values
// of magnitude 2^-11 .. 4.2e6; smaller ones keep an absolute error below
// 2^-18).  The prepacked scales carry the 2^6 that undoes it and the 1/16 of
// the rows whose codes enter the MMA sixteen times larger (see the fold):
// a tile stores s' = 64 s for row gq and s' = 64 s / f for row gq + 8
// (f = 16 at 4 bits, 1 at 8 bits), scaled by powers of two, so exactly.
constexpr float X_SCALE = 0.015625f;
constexpr float S_ROW0 = 64.f;                               // row gq
template <int BITS> constexpr float S_ROW1 = BITS == 4 ? 4.f : 64.f;  // row gq + 8

// bf16 bits of (bf16 value) * 2^j: the same significand, so exact (up to
// overflow to infinity, as the product in fp32 would overflow too).
__device__ __forceinline__ uint32_t bf16_pow2_scaled(uint32_t bits, float pow2) {
  return __float_as_uint(__uint_as_float(bits << 16) * pow2) >> 16;
}
static_assert(Pack<4>::GB == GB_BYTES, "4-bit layout");
// group-blocks per stage: 16 (72 KB), or 12 / 8 where a larger activation
// window is worth more than fewer, larger stages; 8-bit group-blocks are
// 8704 B, so 8 or 4 of them (70 KB or 35 KB).  Every option is a multiple
// of the four warps that split a stage's groups.
constexpr int SG_OPTIONS[3] = {16, 12, 8};
constexpr int SG_OPTIONS8[2] = {8, 4};
constexpr int MAX_STAGES = 8;
constexpr int MIN_STAGES = 2;
constexpr int BAR_BYTES = 1024;
constexpr int PART_FLOATS = 4;       // partial floats per lane and warp (at M > 8)

struct Plan {
  int NT;          // 16-row tiles
  int NB;          // batches of 8 tiles
  int G;           // groups per row
  int W;           // group-blocks = NB * G
  int ctas;
  int full_k;      // 1: a CTA whose range covers a whole row may hold all G groups
  int XG;          // window capacity in groups
  int XS;          // activation row stride in shared memory (bytes)
  int nst;         // ring stages
  int xrows;       // activation rows kept in shared memory (M, plus a zero row)
  int red_bytes;   // shared-memory area where the warps of a tile pair add their sums
  int sg;          // group-blocks per stage
  int stage_bytes;
  int aligned;     // 1: CTA ranges hold whole batches (no cross-CTA merge)
  int cl;          // >= 2: each batch is shared by a cluster of cl CTAs (0: no cluster)
  int sp;          // >= 2: each batch is split over sp CTAs, merged in global memory (0: no split)
  int gb_bytes;    // bytes of one group-block (4-bit 4608, 8-bit 8704)
  int stall;       // test aid: arm the first weight copy without issuing it (waits run out)
};

// Shared memory: barriers, ring, the warps' reduction area, activation rows
// of the window (+ one row of zeros for the padding lanes), and the window's
// per-group activation sums.
static size_t fixed_bytes(int xrows, int XG, int red_bytes) {
  return (size_t)BAR_BYTES + (size_t)red_bytes + (size_t)xrows * (XG * 128 + 16) +
         (size_t)XG * 16 * sizeof(float) + 1024;
}
static size_t smem_fixed(const Plan &p) { return fixed_bytes(p.xrows, p.XG, p.red_bytes); }
static size_t smem_bytes(const Plan &p) { return smem_fixed(p) + (size_t)p.nst * p.stage_bytes; }

// Rows are padded by 16 bytes (stride = 16 mod 128) so the per-lane 16-byte
// fragment loads are free of bank conflicts.
static Plan make_plan(int N, int K, int H, int M, int sms, int smem_optin, int bits = 4,
                      int cl_max = 0, bool split = false) {
  Plan p{};
  p.gb_bytes = bits == 8 ? Pack<8>::GB : Pack<4>::GB;
  p.NT = (N + TILE_N - 1) / TILE_N;
  p.NB = (p.NT + BATCH - 1) / BATCH;
  p.G = K / GROUP;
  const long long W = (long long)p.NB * p.G;
  p.W = (int)std::min<long long>(W, 0x7fffffffLL);
  p.ctas = (int)std::min<long long>(W, sms);
  // With at least one batch per CTA, the ranges hold whole batches: a CTA
  // streams at most one batch more than the mean, and no batch is cut, so
  // nothing is merged across CTAs (no partial sums, no arrival handshake at
  // the end of the launch).  At 1.8 batches per CTA (gate+up on 152 SMs)
  // that is 7% faster than the even stream-K split with its merges; with
  // fewer batches than CTAs the split keeps every SM streaming.
  p.aligned = p.NB >= p.ctas ? 1 : 0;
  // With fewer batches than SMs, a thread-block cluster of cl CTAs takes each
  // batch: its CTAs split the batch's groups and add their partial sums in
  // distributed shared memory at a cluster barrier.  Nothing is merged through
  // global memory (no partial slots, no arrival atomics, no release fences),
  // which is what a batch cut between CTAs costs in the stream-K split.
  // It pays where the SMs it leaves idle cost less than the merges it saves:
  // a CTA consumes a group-block in about 0.11 us and a cut batch costs it
  // about 1.5 us, so at most 14 group-blocks more per CTA than the even split
  // (the o projection, 40 batches x 3 CTAs, qualifies; down, with 91 instead
  // of 72 group-blocks per CTA, does not).
  p.cl = 0;
  if (cl_max >= 2 && !p.aligned) {
    const int cl = std::min(std::min(std::min(8, cl_max), sms / p.NB), p.G);
    const long long ctas = (long long)p.NB * cl;
    if (cl >= 2 && W * (sms - ctas) < 14LL * ctas * sms) {
      p.cl = cl;
      p.ctas = (int)ctas;
    }
  }
  // Without a cluster, each batch may still be split over sp CTAs whose
  // ranges stay inside it: every CTA then holds one segment, and the batch is
  // merged by its last CTA to arrive.  A range of the even split that crosses
  // a batch boundary costs its CTA about 1 us more at the end (two batches'
  // partials and, usually, a merge), so the split pays for at most 9
  // group-blocks more per CTA (qkv: 48 batches x 3 CTAs, 26.7 instead of
  // 25.3 group-blocks).
  p.sp = 0;
  if (split && !p.aligned && !p.cl) {
    const int sp = std::min(std::min(8, sms / p.NB), p.G);
    const long long ctas = (long long)p.NB * sp;
    if (sp >= 2 && W * (sms - ctas) < 9LL * ctas * sms) {
      p.sp = sp;
      p.ctas = (int)ctas;
    }
  }
  p.xrows = M + (M < 8 * H ? 1 : 0);
  p.red_bytes = CWARPS * 32 * TPW * H * 4 * (int)sizeof(float);
  const long long budget = (long long)smem_optin - 2048;  // static smem and slack
  // For each stage size, the widest window that still leaves MIN_STAGES ring
  // stages.  Take the largest stage size whose window holds min(G, 80)
  // groups, else the one with the widest window.
  const int want = std::min(p.G, 80);
  int best_sg = 0, best_xg = 0;
  const int nopt = bits == 8 ? 2 : 3;
  for (int oi = 0; oi < nopt; ++oi) {
    const int sg = bits == 8 ? SG_OPTIONS8[oi] : SG_OPTIONS[oi];
    int XG = want;
    for (; XG > 8; XG -= 8) {
      const long long fixed = (long long)fixed_bytes(p.xrows, XG, p.red_bytes);
      if (budget - fixed >= (long long)MIN_STAGES * sg * p.gb_bytes) break;
    }
    if (XG > best_xg) {
      best_xg = XG;
      best_sg = sg;
    }
    if (XG >= want) break;
  }
  p.sg = best_sg;
  p.stage_bytes = best_sg * p.gb_bytes;
  p.XG = best_xg;
  p.XS = p.XG * 128 + 16;
  p.full_k = p.G <= p.XG;
  const long long room = budget - (long long)smem_fixed(p);
  p.nst = (int)std::max<long long>(2, std::min<long long>(MAX_STAGES, room / p.stage_bytes));
  return p;
}

// Workspace: per-batch arrival counters, then two partial slots per CTA
// (its first and last batch segment), each 16 warps x 32 lanes x 4 floats.
// one arrival counter per 128-byte line (CTAs of different batches arrive
// at the same moment; a shared line would serialise their atomics)
constexpr int CSTRIDE = 32;
static size_t counters_bytes(const Plan &p) { return ((size_t)p.NB * 4 * CSTRIDE + 255) / 256 * 256; }
static size_t workspace_bytes(const Plan &p) {
  return counters_bytes(p) + (size_t)2 * p.ctas * CWARPS * 32 * PART_FLOATS * sizeof(float);
}
static int smem_optin() {
  static int v = 0;
  if (!v) {
    int d = 0, x = 0;
    if (cudaGetDevice(&d) == cudaSuccess &&
        cudaDeviceGetAttribute(&x, cudaDevAttrMaxSharedMemoryPerBlockOptin, d) == cudaSuccess)
      v = x;
    else
      return 227 * 1024;
  }
  return v;
}

// ----------------------------------------------------------- prepack ---
// One thread per (tile, group, lane).  For k16 step s of the group, lane
// (gq = lane/4, tq = lane%4) holds one word whose nibble j is the code of
//   row gq + 8*(j&1),  k = 16*tq + 4*s + 2*((j>>1)&1) + ((j>>2)&1)
// so that (w >> 4i) & 0x000F000F is MMA A-fragment register i.  The MMA's
// logical k order is thereby permuted within the group so that the B fragment
// of step s is the four activations x[16tq+4s .. 16tq+4s+3]: each lane's B
// fragments for the whole group are 32 contiguous bytes of the activation row.
// Tile t of batch b = t/8 lands at ((b*G + g)*8 + t%8)*576.
__global__ void prepack_kernel(const uint32_t *__restrict__ wq, const uint16_t *__restrict__ sc,
                               const uint16_t *__restrict__ bi, int N, int K, int NTP, int G,
                               uint8_t *__restrict__ out) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)NTP * G * 32) return;
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
  const int b = t / BATCH, jt = t % BATCH;
  uint8_t *blk = out + (((size_t)b * G + g) * BATCH + jt) * BLOCK_BYTES;
  *reinterpret_cast<uint4 *>(blk + lane * 16) = make_uint4(words[0], words[1], words[2], words[3]);
  if (tq == 0) {
    const int n0 = TILE_N * t + gq, n1 = n0 + 8;
    const uint32_t s0 = n0 < N ? bf16_pow2_scaled(sc[(size_t)n0 * G + g], S_ROW0) : 0u;
    const uint32_t s1 = n1 < N ? bf16_pow2_scaled(sc[(size_t)n1 * G + g], S_ROW1<4>) : 0u;
    const uint32_t b0 = n0 < N ? bi[(size_t)n0 * G + g] : 0u;
    const uint32_t b1 = n1 < N ? bi[(size_t)n1 * G + g] : 0u;
    *reinterpret_cast<uint2 *>(blk + CODE_BYTES + gq * 8) =
        make_uint2(s0 | (s1 << 16), b0 | (b1 << 16));
  }
}

// 8-bit codes: the same (row, k) positions per lane and k16 step as above,
// one byte per code, in two words per step.  Word x (0, 1) of step s holds
//   byte j: row gq + 8*(j&1),  k = 16*tq + 4*s + 2*x + ((j>>1)&1)
// so that bytes 0 and 2 of a word are one A-fragment register's pair of
// codes and bytes 1 and 3 the next one's: w & 0x00FF00FF and
// (w >> 8) & 0x00FF00FF, or-ed into the fp16 bits 0x6400, are 1024 + q.
// Steps 0-1 of every lane form the first 512 bytes of the tile's codes,
// steps 2-3 the second (16 contiguous bytes per lane in each half).
__global__ void prepack8_kernel(const uint32_t *__restrict__ wq, const uint16_t *__restrict__ sc,
                                const uint16_t *__restrict__ bi, int N, int K, int NTP, int G,
                                uint8_t *__restrict__ out) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)NTP * G * 32) return;
  const int lane = (int)(idx & 31);
  const long long tg = idx >> 5;
  const int g = (int)(tg % G);
  const int t = (int)(tg / G);
  const int gq = lane >> 2, tq = lane & 3;
  const int KW = K / 4;
  uint32_t words[8];
#pragma unroll
  for (int s = 0; s < 4; ++s)
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      uint32_t w = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int row = gq + ((j & 1) ? 8 : 0);
        const int kk = 16 * tq + 4 * s + 2 * x + ((j >> 1) & 1);
        const int n = TILE_N * t + row;
        const int k = GROUP * g + kk;
        uint32_t code = 0;
        if (n < N) code = (wq[(size_t)n * KW + (k >> 2)] >> (8 * (k & 3))) & 255u;
        w |= code << (8 * j);
      }
      words[2 * s + x] = w;
    }
  const int b = t / BATCH, jt = t % BATCH;
  uint8_t *blk = out + (((size_t)b * G + g) * BATCH + jt) * Pack<8>::BLOCK;
  *reinterpret_cast<uint4 *>(blk + lane * 16) = make_uint4(words[0], words[1], words[2], words[3]);
  *reinterpret_cast<uint4 *>(blk + CODE_BYTES + lane * 16) =
      make_uint4(words[4], words[5], words[6], words[7]);
  if (tq == 0) {
    const int n0 = TILE_N * t + gq, n1 = n0 + 8;
    const uint32_t s0 = n0 < N ? bf16_pow2_scaled(sc[(size_t)n0 * G + g], S_ROW0) : 0u;
    const uint32_t s1 = n1 < N ? bf16_pow2_scaled(sc[(size_t)n1 * G + g], S_ROW1<8>) : 0u;
    const uint32_t b0 = n0 < N ? bi[(size_t)n0 * G + g] : 0u;
    const uint32_t b1 = n1 < N ? bi[(size_t)n1 * G + g] : 0u;
    *reinterpret_cast<uint2 *>(blk + Pack<8>::CODE + gq * 8) =
        make_uint2(s0 | (s1 << 16), b0 | (b1 << 16));
  }
}

// ------------------------------------------------------------- kernel ---
struct Smem {
  uint64_t *full, *empty, *xfull, *xempty;
  uint64_t *seg1, *seg1_arr;  // first segment's partial stored; its arrival made
  uint8_t *ring, *xraw;
  float *red, *xs;
  uint32_t ring_a, xraw_a, xs_a;  // shared-space addresses
};

__device__ __forceinline__ Smem carve(uint8_t *base, const Plan &p) {
  Smem s;
  s.full = reinterpret_cast<uint64_t *>(base);
  s.empty = s.full + MAX_STAGES;
  s.xfull = s.empty + MAX_STAGES;
  s.xempty = s.xfull + 1;
  s.seg1 = s.xempty + 1;
  s.seg1_arr = s.seg1 + 1;
  s.ring = base + BAR_BYTES;
  s.red = reinterpret_cast<float *>(s.ring + (size_t)p.nst * p.stage_bytes);
  s.xraw = s.ring + (size_t)p.nst * p.stage_bytes + p.red_bytes;
  s.xs = reinterpret_cast<float *>(s.xraw + (size_t)p.xrows * p.XS);
  s.ring_a = smem_u32(s.ring);
  s.xraw_a = smem_u32(s.xraw);
  s.xs_a = smem_u32(s.xs);
  return s;
}

// A lane of warp (pair, rr) finishes ES of its pair's accumulator floats:
// e = rr*ES + i, laid out as tile tt = e / (4H), row half h = (e/4) % H and
// m16n8 accumulator register j = e % 4.
template <int H, int ES>
__device__ __forceinline__ void store_share(void *y, int y_f32, int M, int N, int tile0, int rr,
                                            int lane, const float (&z)[ES]) {
  const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
  for (int i = 0; i < ES; ++i) {
    const int e = rr * ES + i;
    const int tt = e / (4 * H), h = (e >> 2) % H, j = e & 3;
    const int n = TILE_N * (tile0 + tt) + gq + ((j & 2) ? 8 : 0);
    const int m = 8 * h + 2 * tq + (j & 1);
    if (m < M && n < N) {
      if (y_f32)
        static_cast<float *>(y)[(size_t)m * N + n] = z[i];
      else
        static_cast<__nv_bfloat16 *>(y)[(size_t)m * N + n] = __float2bfloat16_rn(z[i]);
    }
  }
}

__device__ __forceinline__ float2 make_vec(const float (&z)[2]) { return make_float2(z[0], z[1]); }
__device__ __forceinline__ float4 make_vec(const float (&z)[4]) {
  return make_float4(z[0], z[1], z[2], z[3]);
}
__device__ __forceinline__ void add_vec(float (&t)[2], float2 v) {
  t[0] += v.x;
  t[1] += v.y;
}
__device__ __forceinline__ void add_vec(float (&t)[4], float4 v) {
  t[0] += v.x;
  t[1] += v.y;
  t[2] += v.z;
  t[3] += v.w;
}

__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned *p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// CTA whose group-block range contains w.
__device__ __forceinline__ int owner(int w, const Plan &p) {
  if (p.sp) {
    // piece k of a batch starts at group floor(k G / sp)
    const int b = w / p.G, g = w - b * p.G;
    return b * p.sp + ((g + 1) * p.sp - 1) / p.G;
  }
  if (p.aligned) return (int)((((long long)(w / p.G) + 1) * p.ctas - 1) / p.NB);
  return (int)((((long long)w + 1) * p.ctas - 1) / p.W);
}
__device__ __forceinline__ int range_start(int c, const Plan &p) {
  const int pieces = p.cl ? p.cl : p.sp;
  if (pieces) return (c / pieces) * p.G + (c % pieces) * p.G / pieces;
  if (p.aligned) return (int)((long long)c * p.NB / p.ctas) * p.G;
  return (int)((long long)c * p.W / p.ctas);
}

// The CTA's stages: runs of <= sg group-blocks inside one batch and one
// activation window, walked incrementally (no division per stage).  The
// producer and every consumer warp walk the same sequence.
struct StageIter {
  int w, w0, w1, wend_win;
  int b, g, G, XG, win, full_k, sg;
  __device__ void init(int a, int e, const Plan &p) {
    w = a;
    w0 = a;
    w1 = e;
    G = p.G;
    XG = p.XG;
    sg = p.sg;
    // all G groups at once only when the range needs them all; otherwise
    // windows over the range's own groups
    full_k = p.full_k && e - a >= p.G;
    b = a / G;
    g = a - b * G;
    win = 0;
    wend_win = full_k ? e : imin(e, a + XG);
  }
  __device__ bool valid() const { return w < w1; }
  __device__ int count() const { return imin(imin(wend_win - w, sg), G - g); }
  __device__ void advance(int cnt) {
    w += cnt;
    g += cnt;
    if (g == G) {
      g = 0;
      ++b;
    }
    if (w == wend_win && w < w1) {
      ++win;
      wend_win = imin(w1, wend_win + XG);
    }
  }
  // window k covers group-blocks [w0 + k*XG, min(w1, w0 + (k+1)*XG)): its
  // groups are a cyclic interval [gstart, gstart + len) modulo G
  __device__ void window_span(int k, int &gstart, int &len) const {
    if (full_k) {
      gstart = 0;
      len = G;
      return;
    }
    const int a = w0 + k * XG;
    gstart = a % G;
    len = imin(w1, a + XG) - a;
  }
};

// Activation window k: TMA copies of the M rows' groups [gstart, gstart+len)
// (cyclic modulo G, so at most two copies per row).
__device__ __forceinline__ void issue_window(const StageIter &it, const Smem &sm, int XS, int k,
                                             const __nv_bfloat16 *__restrict__ x, int M, int K,
                                             uint64_t pol) {
  int gstart, len;
  it.window_span(k, gstart, len);
  const int first = imin(len, it.G - gstart);
  mbar_arrive_expect_tx(sm.xfull, (uint32_t)(M * len * 128));
  for (int m = 0; m < M; ++m) {
    const __nv_bfloat16 *row = x + (size_t)m * K;
    tma_load_1d(sm.xraw + (size_t)m * XS, row + (size_t)gstart * GROUP, (uint32_t)(first * 128),
                sm.xfull, pol);
    if (len > first)
      tma_load_1d(sm.xraw + (size_t)m * XS + (size_t)first * 128, row, (uint32_t)((len - first) * 128),
                  sm.xfull, pol);
  }
}

// One group of the stage for this warp's two tiles: the activation fragments
// and group sums are loaded once and shared by both tiles.
template <int H, int BITS>
__device__ __forceinline__ void consume_group(uint32_t blk, uint32_t xl0, uint32_t xl1, uint32_t xsl,
                                              int lane, int gq, float (&yv)[TPW][H][4]) {
  using PK = Pack<BITS>;
  uint4 xa[H], xb[H];
  xa[0] = lds128(xl0);
  xb[0] = lds128(xl0 + 16);
  if (H == 2) {
    xa[H - 1] = lds128(xl1);
    xb[H - 1] = lds128(xl1 + 16);
  }
  float xs0[H], xs1[H];
#pragma unroll
  for (int h = 0; h < H; ++h) {
    const uint2 v = lds64(xsl + (uint32_t)(8 * h * 4));
    xs0[h] = __uint_as_float(v.x);
    xs1[h] = __uint_as_float(v.y);
  }
#pragma unroll
  for (int tt = 0; tt < TPW; ++tt) {
    const uint4 wv = lds128(blk + tt * PK::BLOCK + lane * 16);
    uint4 wv2 = wv;
    if (BITS == 8) wv2 = lds128(blk + tt * PK::BLOCK + CODE_BYTES + lane * 16);
    const uint2 sb = lds64(blk + tt * PK::BLOCK + PK::CODE + gq * 8);
    float acc[H][4];
#pragma unroll
    for (int st4 = 0; st4 < 4; ++st4) {
      uint32_t a0, a1, a2, a3;
      if (BITS == 4) {
        // fp16 0x6400 | c is 1024 + c exactly and 0x6400 | (c << 4) is
        // 1024 + 16c: the row-gq codes (nibbles 0, 2, 4, 6) in place, the
        // row-gq+8 codes (nibbles 1, 3, 5, 7) sixteen times larger, which the
        // fold undoes per output row
        const uint32_t w = st4 == 0 ? wv.x : st4 == 1 ? wv.y : st4 == 2 ? wv.z : wv.w;
        const uint32_t w8 = w >> 8;
        a0 = and_or<0x000F000Fu, 0x64006400u>(w);
        a1 = and_or<0x00F000F0u, 0x64006400u>(w);
        a2 = and_or<0x000F000Fu, 0x64006400u>(w8);
        a3 = and_or<0x00F000F0u, 0x64006400u>(w8);
      } else {
        // a whole byte per fp16 register: 0x6400 | q is 1024 + q exactly
        const uint4 &wsrc = st4 < 2 ? wv : wv2;
        const uint32_t wa = (st4 & 1) ? wsrc.z : wsrc.x;
        const uint32_t wb = (st4 & 1) ? wsrc.w : wsrc.y;
        a0 = and_or<0x00FF00FFu, 0x64006400u>(wa);
        a1 = and_or<0x00FF00FFu, 0x64006400u>(wa >> 8);
        a2 = and_or<0x00FF00FFu, 0x64006400u>(wb);
        a3 = and_or<0x00FF00FFu, 0x64006400u>(wb >> 8);
      }
#pragma unroll
      for (int h = 0; h < H; ++h) {
        const uint4 &xv = (st4 < 2) ? xa[h] : xb[h];
        const uint32_t b0 = (st4 & 1) ? xv.z : xv.x;
        const uint32_t b1 = (st4 & 1) ? xv.w : xv.y;
        if (st4 == 0)
          mma_f16_16816_zc(acc[h], a0, a1, a2, a3, b0, b1);
        else
          mma_f16_16816(acc[h], a0, a1, a2, a3, b0, b1);
      }
    }
    // acc = 2^-6 * sum_k x (1024 + f q) with f = 1 (row gq; both rows at 8
    // bits) or 16 (row gq+8 at 4 bits), so with the prepacked s' = 64 s / f
    //   sum_k x (s q + b) = s' acc + (b - 16 s') sum_k x
    const float sa0 = bf16lo(sb.x), sa1 = bf16hi(sb.x);
    const float c0 = fmaf(-16.f, sa0, bf16lo(sb.y));
    const float c1 = fmaf(-16.f, sa1, bf16hi(sb.y));
#pragma unroll
    for (int h = 0; h < H; ++h) {
      yv[tt][h][0] = fmaf(sa0, acc[h][0], fmaf(c0, xs0[h], yv[tt][h][0]));
      yv[tt][h][1] = fmaf(sa0, acc[h][1], fmaf(c0, xs1[h], yv[tt][h][1]));
      yv[tt][h][2] = fmaf(sa1, acc[h][2], fmaf(c1, xs0[h], yv[tt][h][2]));
      yv[tt][h][3] = fmaf(sa1, acc[h][3], fmaf(c1, xs1[h], yv[tt][h][3]));
    }
  }
}

__device__ __forceinline__ float lds32f(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// CUDA-core comparison path (MR = M activation rows, M <= 8 half only): the
// same group of this warp's two tiles as consume_group, with every code
// converted to fp32 ((q | 0x4B000000) - 2^23, exact) and multiplied into
// per-lane fp32 accumulators with FFMA instead of the tensor-core MMA.  The
// lane covers its 16 k of the group for rows gq and gq+8; the four lanes of
// a row are added at the end of the batch segment, and the bias term b * sum x
// is added once (by the lane with tq = 0).
template <int MR>
__device__ __forceinline__ void consume_group_fma(uint32_t blk, uint32_t xr0, int XS, uint32_t xsl,
                                                  int lane, int gq, int tq,
                                                  float (&yf)[TPW][2][MR]) {
  uint4 wv[TPW];
  uint2 sb[TPW];
#pragma unroll
  for (int tt = 0; tt < TPW; ++tt) {
    wv[tt] = lds128(blk + tt * BLOCK_BYTES + lane * 16);
    sb[tt] = lds64(blk + tt * BLOCK_BYTES + CODE_BYTES + gq * 8);
  }
  float acc[TPW][2][MR];
#pragma unroll
  for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
    for (int nn = 0; nn < 2; ++nn)
#pragma unroll
      for (int m = 0; m < MR; ++m) acc[tt][nn][m] = 0.f;
#pragma unroll
  for (int st4 = 0; st4 < 4; ++st4) {
    float xv[MR][4];  // x[m][16 tq + 4 st4 + 0..3]
#pragma unroll
    for (int m = 0; m < MR; ++m) {
      const uint2 v = lds64(xr0 + (uint32_t)(m * XS) + 8 * st4);  // fp16 x * 2^-6
      xv[m][0] = f16lo(v.x) * (1.f / X_SCALE);
      xv[m][1] = f16hi(v.x) * (1.f / X_SCALE);
      xv[m][2] = f16lo(v.y) * (1.f / X_SCALE);
      xv[m][3] = f16hi(v.y) * (1.f / X_SCALE);
    }
#pragma unroll
    for (int tt = 0; tt < TPW; ++tt) {
      const uint32_t w = st4 == 0 ? wv[tt].x : st4 == 1 ? wv[tt].y : st4 == 2 ? wv[tt].z : wv[tt].w;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float q = __uint_as_float(((w >> (4 * j)) & 15u) | 0x4B000000u) - 8388608.0f;
        const int nn = j & 1, kk = 2 * ((j >> 1) & 1) + ((j >> 2) & 1);
#pragma unroll
        for (int m = 0; m < MR; ++m) acc[tt][nn][m] = fmaf(q, xv[m][kk], acc[tt][nn][m]);
      }
    }
  }
  float xsm[MR];
#pragma unroll
  for (int m = 0; m < MR; ++m) xsm[m] = tq == 0 ? lds32f(xsl + 4 * m) : 0.f;
#pragma unroll
  for (int tt = 0; tt < TPW; ++tt) {
    const float sc[2] = {bf16lo(sb[tt].x) * (1.f / S_ROW0), bf16hi(sb[tt].x) * (1.f / S_ROW1<4>)};
    const float bc[2] = {bf16lo(sb[tt].y), bf16hi(sb[tt].y)};
#pragma unroll
    for (int nn = 0; nn < 2; ++nn)
#pragma unroll
      for (int m = 0; m < MR; ++m)
        yf[tt][nn][m] = fmaf(sc[nn], acc[tt][nn][m], fmaf(bc[nn], xsm[m], yf[tt][nn][m]));
  }
}

// ------------------------------------------------- top-k lists epilogue ---
// The lm_head launch can end with the first stage of the acceptance: every
// CTA, holding whole batches, selects per logits row the top-k of its own
// vocabulary range (every logit equal to the k-th largest kept) and writes
// it as a short list; the acceptance merges the CTAs' lists instead of
// scanning the logits again.
constexpr int LISTS_HDR = 64;  // header: M, ctas, cap, k, N
struct TopkOut {
  uint8_t *lists;  // null: no lists
  int k;           // top-k per row (1 at temperature 0)
  int cap;         // entries per list: the largest CTA range
};
__host__ __device__ inline size_t list_stride(int cap) { return 16 + (size_t)cap * 8; }

// Order-preserving integer image of a logit (NaN excluded, -0 = +0).
__device__ __forceinline__ uint32_t logit_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Rows of the CTA's columns [c0, c1) of y, in groups of NW warps (one named
// barrier per group, ids 2..): per row, every warp takes the top-k (ties
// kept) of its slice of the columns, and one warp takes the exact top-k of
// those candidates -- the CTA's top-k -- into the list.  Per group the
// scratch holds the row's keys, the candidates (key, column) and a counter:
// 12 bytes per column of the range plus 16.
__host__ __device__ inline size_t topk_scratch(int cap) { return (size_t)cap * 12 + 16; }

template <int NW>
__device__ void topk_lists(const float *y, int M, int N, int c0, int c1, const TopkOut &to,
                           int ctas, int cta, uint8_t *scr, int ctid) {
  constexpr int GT = NW * 32;                // threads per group
  constexpr int NG = CWARPS / NW;            // groups
  const int grp = ctid / GT, gt = ctid % GT, lane = ctid & 31, wig = gt >> 5;
  const int bar = 2 + grp;
  const int n = c1 - c0;
  uint32_t *keys = reinterpret_cast<uint32_t *>(scr + (size_t)grp * topk_scratch(to.cap));
  uint32_t *ckey = keys + to.cap, *ccol = ckey + to.cap;
  int *cnt = reinterpret_cast<int *>(ccol + to.cap);
  const int seg = (n + NW - 1) / NW;         // columns per warp
  const int s0 = imin(n, wig * seg), s1 = imin(n, s0 + seg);
  const unsigned lt = (1u << lane) - 1u;
  for (int m = grp; m < M; m += NG) {
    const float *yr = y + (size_t)m * N + c0;
    for (int i = s0 + lane; i < s1; i += 32) keys[i] = logit_key(__ldcg(yr + i));
    if (gt == 0) *cnt = 0;
    named_barrier(bar, GT);
    // this warp's top-k of its slice: candidates of the CTA's top-k
    const uint32_t tw = warp_kth_largest(keys + s0, s1 - s0, to.k);
    for (int base = s0; base < s1; base += 32) {
      const int i = base + lane;
      const bool keep = i < s1 && keys[i] >= tw;
      const unsigned msk = __ballot_sync(0xffffffffu, keep);
      if (msk) {
        const int leader = __ffs(msk) - 1;
        int pos = 0;
        if (lane == leader) pos = atomicAdd(cnt, __popc(msk));
        pos = __shfl_sync(0xffffffffu, pos, leader) + __popc(msk & lt);
        if (keep) {
          ckey[pos] = keys[i];
          ccol[pos] = (uint32_t)(c0 + i);
        }
      }
    }
    named_barrier(bar, GT);
    if (wig == 0) {
      const int nc = *cnt;
      const uint32_t t = warp_kth_largest(ckey, nc, to.k);
      uint8_t *L = to.lists + LISTS_HDR + ((size_t)m * ctas + cta) * list_stride(to.cap);
      uint32_t *lk = reinterpret_cast<uint32_t *>(L + 16), *li = lk + to.cap;
      int w = 0;
      for (int base = 0; base < nc; base += 32) {
        const int i = base + lane;
        const bool keep = i < nc && ckey[i] >= t;
        const unsigned msk = __ballot_sync(0xffffffffu, keep);
        if (keep) {
          lk[w + __popc(msk & lt)] = ckey[i];
          li[w + __popc(msk & lt)] = ccol[i];
        }
        w += __popc(msk);
      }
      if (lane == 0) *reinterpret_cast<int *>(L) = w;
    }
    named_barrier(bar, GT);  // keys, candidates and the counter are reused
  }
}

// FM = 0: tensor-core MMA; FM = MR > 0: the CUDA-core comparison path for M = MR
// (4-bit codes only).  BITS: 4 or 8.
// TOPK: the top-k lists epilogue (whole batches per CTA, fp32 output).
template <int H, int SG, int FM, int BITS = 4, int TOPK = 0>
__global__ void __launch_bounds__(THREADS, 1)
    qmm_kernel(const __nv_bfloat16 *__restrict__ x, const uint8_t *__restrict__ packed, void *y,
               int y_f32, int M, int N, int K, Plan plan, float *__restrict__ part,
               unsigned *__restrict__ counters, unsigned *err, TopkOut topk) {
  static_assert(BITS == 4 || FM == 0, "the CUDA-core path reads 4-bit codes");
  constexpr int GBB = Pack<BITS>::GB;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int nst = plan.nst;
  const Smem sm = carve(base, plan);
  const int XS = plan.XS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int G = plan.G;
  const int cta = blockIdx.x;
  const int w0 = range_start(cta, plan), w1 = range_start(cta + 1, plan);
  __shared__ int s_last, s_last2;

  if (tid == 0) {
    for (int i = 0; i < nst; ++i) {
      mbar_init(&sm.full[i], 1);
      mbar_init(&sm.empty[i], CWARPS);
    }
    mbar_init(sm.xfull, 1);
    mbar_init(sm.xempty, CWARPS);
    mbar_init(sm.seg1, CWARPS);
    mbar_init(sm.seg1_arr, 1);
    fence_barrier_init();
  }
  // the zero row (padding lanes read it) and the padding rows' group sums
  if (plan.xrows > M)
    for (int i = tid; i < XS / 16; i += THREADS)
      *reinterpret_cast<uint4 *>(sm.xraw + (size_t)M * XS + i * 16) = make_uint4(0u, 0u, 0u, 0u);
  for (int i = tid; i < plan.XG * 16; i += THREADS)
    if ((i & 15) >= M) sm.xs[i] = 0.f;
  __syncthreads();
  pdl_launch_dependents();

  // A range of the stream-K plan that starts inside a batch and reaches into
  // the next one holds a cut first segment: its partial is stored when the
  // batch changes, and its arrival is made here, off the consumers' path.
  const bool cut_first = !plan.aligned && !plan.cl && w0 < w1 && w0 % G != 0 && (w1 - 1) / G != w0 / G;
  if (warp == CWARPS + 1) {
    // -------------------------------------------------------- arrivals --
    if (lane == 0 && cut_first) {
      int last = 0;
      if (spin_wait(sm.seg1, 0u, err)) {
        // acquire-release arrival: the consumers' partial stores precede
        // their mbarrier arrivals (release, CTA scope), which this wait
        // acquires before the release at GPU scope
        const int b = w0 / G;
        const int c_first = owner(b * G, plan), c_last = owner(b * G + G - 1, plan);
        unsigned *ctr = counters + (size_t)b * CSTRIDE;
        const unsigned prev = atom_add_acq_rel_gpu(ctr, 1u);
        last = prev == (unsigned)(c_last - c_first);
        if (last) *ctr = 0u;  // ready for the next call
      }
      s_last = last;
      mbar_arrive(sm.seg1_arr);  // (release: s_last to the consumers)
    }
    __syncwarp();
    if (plan.cl) {
      // every thread meets the consumers' two cluster barriers
      cluster_sync_all();
      cluster_sync_all();
    }
    return;
  }

  if (warp == CWARPS) {
    // ------------------------------------------------------- producer --
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      StageIter it;
      it.init(w0, w1, plan);
      bool ok = true;
      uint32_t q = 0, slot = 0, phase = 1;
      // window 0 comes from consumer warp 0 as soon as the predecessor grid
      // has completed; the weights do not depend on it and stream from the start
      int x_issued = 1;
      while (it.valid() && ok) {
        // Wait for a free ring slot.  Meanwhile issue the activation window of
        // the stages in flight as soon as it may be loaded: window k once the
        // consumers have left window k-1.  Weights keep streaming across
        // window boundaries.
        const long long t0 = clock64();
        for (;;) {
          if (x_issued <= it.win) {
            const bool ready = mbar_test_wait(sm.xempty, (uint32_t)(x_issued - 1) & 1u);
            if (ready) {
              issue_window(it, sm, XS, x_issued, x, M, K, pol);
              ++x_issued;
              continue;
            }
            if (mbar_test_wait(&sm.empty[slot], phase)) break;
            __nanosleep(64);  // poll both barriers without taking the consumers' issue slots
          } else if (mbar_try_wait(&sm.empty[slot], phase)) {
            break;  // (try_wait suspends the thread until the phase completes or a time limit)
          }
          if (clock64() - t0 > WAIT_LIMIT_CYCLES) {
            atomicOr(err, ERR_TIMEOUT);
            ok = false;
            break;
          }
        }
        if (!ok) break;
        const int cnt = it.count();
        mbar_arrive_expect_tx(&sm.full[slot], (uint32_t)(cnt * GBB));
        if (!(plan.stall && q == 0))
          tma_load_1d(sm.ring + (size_t)slot * (SG * GBB), packed + (size_t)it.w * GBB,
                      (uint32_t)(cnt * GBB), &sm.full[slot], pol);
        it.advance(cnt);
        ++q;
        if (++slot == (uint32_t)nst) {
          slot = 0;
          phase ^= 1u;
        }
      }
      // windows not issued yet: all of them when the range is shorter than the
      // ring, and the last ones
      while (ok && x_issued <= it.win) {
        if (!(ok = spin_wait(sm.xempty, (uint32_t)(x_issued - 1) & 1u, err))) break;
        issue_window(it, sm, XS, x_issued, x, M, K, pol);
        ++x_issued;
      }
      if (!ok) {
        // Drain: do not leave while copies may still land in shared memory.
        const uint32_t first = q > (uint32_t)nst ? q - nst : 0u;
        for (uint32_t qq = first; qq < q; ++qq) mbar_wait(&sm.full[qq % nst], (qq / nst) & 1, err);
        if (x_issued > 0) mbar_wait(sm.xfull, (uint32_t)(x_issued - 1) & 1u, err);
      }
    }
    __syncwarp();
    if (plan.cl) {
      // the consumers' two cluster barriers (partials written; partials read)
      cluster_sync_all();
      cluster_sync_all();
    }
    return;
  }

  // ------------------------------------------------------- consumers --
  pdl_wait();  // activations, outputs and workspace follow the predecessor
  if (warp == 0 && lane == 0 && w0 < w1) {
    // the first activation window, not queued behind the ring's weights
    StageIter it0;
    it0.init(w0, w1, plan);
    issue_window(it0, sm, XS, 0, x, M, K, l2_evict_first_policy());
  }
  const int gq = lane >> 2, tq = lane & 3;
  // this lane's activation row in each n8 half (padding rows read zeros)
  const int r0 = gq < M ? gq : M, r1 = 8 + gq < M ? 8 + gq : M;
  // (the tile-pair warps' group residue rr is folded into the bases)
  const uint32_t xlane0 = sm.xraw_a + (uint32_t)(r0 * XS + 32 * tq + (warp / PAIRS) * 128);
  const uint32_t xlane1 = sm.xraw_a + (uint32_t)(r1 * XS + 32 * tq + (warp / PAIRS) * 128);
  const uint32_t xslane = sm.xs_a + (uint32_t)(2 * tq * 4 + (warp / PAIRS) * 64);
  const int pr = warp % PAIRS, rr = warp / PAIRS;  // tile pair, group residue
  const uint32_t wbase = (uint32_t)(pr * TPW * Pack<BITS>::BLOCK + rr * GBB);
  bool ok = true;
  int cur_win = -1, wgstart = 0;
  int cur_b = -1, seg_lo = 0, seg_hi = 0;
  bool first_seg = true;
  float yv[TPW][H][4];
  // CUDA-core comparison path: per-lane accumulators and row-0 bases
  constexpr int MRF = FM > 0 ? FM : 1;
  float yf[TPW][2][MRF];
  const uint32_t xr0 = sm.xraw_a + (uint32_t)(32 * tq + (warp / PAIRS) * 128);
  const uint32_t xsf = sm.xs_a + (uint32_t)((warp / PAIRS) * 64);

  // End of a batch segment.  The GSPLIT warps of a tile pair hold sums over
  // different groups: reduce() adds them in shared memory in warp order,
  // each warp finishing ES floats per lane.  A whole batch is then stored
  // directly.  A cut batch (stream-K plan) goes to this CTA's partial slot
  // for it, and the last CTA of the batch to arrive adds the slots in CTA
  // order; the arrivals wait until the CTA's work is done, so the
  // mid-range batch change costs no release fence or atomic round trip.
  // Under the cluster plan the cluster's CTAs add their sums through
  // distributed shared memory.
  constexpr int E = TPW * H * 4;   // accumulator floats per lane
  constexpr int ES = E / GSPLIT;   // floats per lane finished by one warp
  static_assert(ES <= PART_FLOATS, "partial slot too small");
  using VecES = typename std::conditional<ES == 4, float4, float2>::type;
  auto reduce = [&](float (&z)[ES]) {
    if (FM > 0) {
      // add the four lanes of each row (fixed butterfly), then take this
      // lane's values in the MMA accumulator layout
#pragma unroll
      for (int tt = 0; tt < TPW; ++tt) {
        float tot[2][MRF];
#pragma unroll
        for (int nn = 0; nn < 2; ++nn)
#pragma unroll
          for (int m = 0; m < MRF; ++m) {
            float v = yf[tt][nn][m];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            tot[nn][m] = v;
          }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int m = 2 * tq + (j & 1);
          float v = 0.f;
#pragma unroll
          for (int mm = 0; mm < MRF; ++mm)
            if (mm == m) v = tot[j >> 1][mm];
          yv[tt][0][j] = v;
        }
      }
    }
    float *red = sm.red;
#pragma unroll
    for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
      for (int h = 0; h < H; ++h)
#pragma unroll
        for (int j = 0; j < 4; ++j) red[(warp * E + (tt * H + h) * 4 + j) * 32 + lane] = yv[tt][h][j];
    named_barrier(1, CWARPS * 32);
#pragma unroll
    for (int i = 0; i < ES; ++i) {
      const int e = rr * ES + i;
      float acc = 0.f;
#pragma unroll
      for (int r2 = 0; r2 < GSPLIT; ++r2) acc += red[((r2 * PAIRS + pr) * E + e) * 32 + lane];
      z[i] = acc;
    }
    named_barrier(1, CWARPS * 32);  // the reduction area is free again
  };
  // partial slot layout: [slot][warp][lane][ES floats]; slot 2*cta for the
  // CTA's first segment, 2*cta + 1 for its last
  auto store_partial = [&](const float (&z)[ES], bool first) {
    const int pslot = 2 * cta + (first ? 0 : 1);
    VecES *pp = reinterpret_cast<VecES *>(part) + ((size_t)pslot * CWARPS + warp) * 32 + lane;
    *pp = make_vec(z);
  };
  // Arrival of this CTA on batch b's counter (one thread, acquire-release:
  // the barrier before it puts the CTA's partial stores ahead of the
  // release, the barrier after it puts the merge's reads behind the acquire).
  auto arrive = [&](int b) -> int {
    const int bw0 = b * G;
    const int c_first = owner(bw0, plan), c_last = owner(bw0 + G - 1, plan);
    unsigned *ctr = counters + (size_t)b * CSTRIDE;
    const unsigned prev = atom_add_acq_rel_gpu(ctr, 1u);
    const int last = prev == (unsigned)(c_last - c_first);
    if (last) *ctr = 0u;  // ready for the next call
    return last;
  };
  // The last CTA of batch b adds the batch's partial slots in CTA order.
  // CTAs after c_first start inside this batch (their first slot); c_first
  // holds it in its first slot only if its range starts at the batch start.
  auto merge = [&](int b) {
    const int bw0 = b * G;
    const int c_first = owner(bw0, plan), c_last = owner(bw0 + G - 1, plan);
    const int nC = c_last - c_first + 1;
    const int ps0 = 2 * c_first + (range_start(c_first, plan) < bw0 ? 1 : 0);
    constexpr int CH = 16 / ES;  // partial loads in flight per lane
    float tot[ES];
#pragma unroll
    for (int i = 0; i < ES; ++i) tot[i] = 0.f;
    const VecES *pbase = reinterpret_cast<const VecES *>(part) + (size_t)warp * 32 + lane;
    for (int i0 = 0; i0 < nC; i0 += CH) {
      VecES v[CH];
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        const int ci = i0 + i;
        const int ps = ci == 0 ? ps0 : 2 * (c_first + ci);
        if (ci < nC) v[i] = __ldcg(pbase + (size_t)ps * CWARPS * 32);
      }
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        if (i0 + i < nC) add_vec(tot, v[i]);
      }
    }
    if (ok) store_share<H, ES>(y, y_f32, M, N, b * BATCH + pr * TPW, rr, lane, tot);
  };
  // Under the cluster plan: this CTA's sums go to its reduction area; after
  // the cluster barrier, CTA rank r adds the cluster's sums for the warps
  // w = r mod cl, in rank order (deterministic), and stores them.  The
  // second barrier keeps every CTA alive until its sums have been read.
  auto cluster_finish = [&](const float (&z)[ES], int b) {
    const uint32_t mine = smem_u32(sm.red) + (uint32_t)((warp * 32 + lane) * ES * sizeof(float));
    *reinterpret_cast<VecES *>(sm.red + (warp * 32 + lane) * ES) = make_vec(z);
    cluster_sync_all();
    if (warp % plan.cl == (int)cluster_ctarank()) {
      float tot[ES];
#pragma unroll
      for (int i = 0; i < ES; ++i) tot[i] = 0.f;
      for (int j = 0; j < plan.cl; ++j) add_vec(tot, ld_cluster(cluster_map(mine, (uint32_t)j), VecES{}));
      if (ok) store_share<H, ES>(y, y_f32, M, N, b * BATCH + pr * TPW, rr, lane, tot);
    }
    cluster_sync_all();
  };
  int pend_b = -1;  // a cut first segment whose arrival waits for the end

  StageIter it;
  it.init(w0, w1, plan);
  uint32_t slot = 0, phase = 0;
  while (it.valid()) {
    const int cnt = it.count();
    const int b = it.b, g = it.g;
    if (it.win != cur_win) {
      if (cur_win >= 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(sm.xempty);  // done with the old activations
      }
      if (ok) ok = spin_wait(sm.xfull, (uint32_t)it.win & 1u, err);
      int len;
      it.window_span(it.win, wgstart, len);
      if (cur_win >= 0) named_barrier(1, CWARPS * 32);  // old group sums no longer read
      // group sums: eight lanes per (row, group), each adding one 16-byte
      // chunk, then a fixed shuffle tree (every quarter-warp reads 128
      // contiguous bytes: no bank conflicts).  Each lane then rewrites its
      // chunk in place as fp16 x * 2^-6, the MMAs' operand type.
      // (row m, group slot sl) = (pi mod M, pi / M); the quotient from a
      // float reciprocal is exact here: pi < 16 * 80 and (pi + 0.5) / M lies
      // at least 1 / 32 away from an integer, far beyond fp32 rounding
      const float inv_m = 1.f / (float)M;
      for (int p0 = warp * 4; p0 < M * len; p0 += CWARPS * 4) {
        const int pi = p0 + (lane >> 3);
        const int sl = (int)(((float)pi + 0.5f) * inv_m), m = pi - sl * M;
        float sum = 0.f;
        if (pi < M * len) {
          const uint32_t ca = sm.xraw_a + (uint32_t)(m * XS + sl * 128 + 16 * (lane & 7));
          const uint4 v = lds128(ca);
          sum = ((bf16lo(v.x) + bf16hi(v.x)) + (bf16lo(v.y) + bf16hi(v.y))) +
                ((bf16lo(v.z) + bf16hi(v.z)) + (bf16lo(v.w) + bf16hi(v.w)));
          uint4 hv;
          hv.x = pack_f16x2(bf16lo(v.x) * X_SCALE, bf16hi(v.x) * X_SCALE);
          hv.y = pack_f16x2(bf16lo(v.y) * X_SCALE, bf16hi(v.y) * X_SCALE);
          hv.z = pack_f16x2(bf16lo(v.z) * X_SCALE, bf16hi(v.z) * X_SCALE);
          hv.w = pack_f16x2(bf16lo(v.w) * X_SCALE, bf16hi(v.w) * X_SCALE);
          sts128(ca, hv);
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        sum += __shfl_xor_sync(0xffffffffu, sum, 4);
        if (pi < M * len && (lane & 7) == 0) sm.xs[sl * 16 + m] = sum;
      }
      named_barrier(1, CWARPS * 32);
      cur_win = it.win;
    }
    if (b != cur_b) {
      if (cur_b >= 0) {
        // the range's first segment (a range holds at most two when it is
        // shorter than a batch; whole batches otherwise)
        float z[ES];
        reduce(z);
        if (seg_lo == 0 && seg_hi == G) {
          if (ok) store_share<H, ES>(y, y_f32, M, N, cur_b * BATCH + pr * TPW, rr, lane, z);
        } else {
          store_partial(z, first_seg);
          pend_b = cur_b;
          __syncwarp();
          if (lane == 0) mbar_arrive(sm.seg1);  // (release: the warp's partial stores)
        }
        first_seg = false;
      }
      cur_b = b;
      seg_lo = g;
#pragma unroll
      for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
        for (int h = 0; h < H; ++h)
#pragma unroll
          for (int j = 0; j < 4; ++j) yv[tt][h][j] = 0.f;
#pragma unroll
      for (int tt = 0; tt < TPW; ++tt)
#pragma unroll
        for (int nn = 0; nn < 2; ++nn)
#pragma unroll
          for (int m = 0; m < MRF; ++m) yf[tt][nn][m] = 0.f;
    }
    if (ok) ok = spin_wait(&sm.full[slot], phase, err);
    if (ok) {
      int xslot = g;
      if (!it.full_k) {
        xslot = g - wgstart;
        if (xslot < 0) xslot += G;
      }
      const uint32_t st = sm.ring_a + slot * (SG * GBB) + wbase;
      const uint32_t xo = (uint32_t)xslot * 128u, xso = (uint32_t)xslot * 64u;
      if (FM > 0) {
        for (int qd = rr; qd < cnt; qd += GSPLIT)
          consume_group_fma<MRF>(st + (qd - rr) * GB_BYTES, xr0 + xo + (uint32_t)(qd - rr) * 128u, XS,
                                 xsf + xso + (uint32_t)(qd - rr) * 64u, lane, gq, tq, yf);
      } else if (H == 1 && cnt == SG) {
        // full stage at M <= 8: this warp's SG / GSPLIT groups at fixed
        // offsets (at M > 8 the unrolled body would not fit the registers)
#pragma unroll
        for (int i = 0; i < SG / GSPLIT; ++i)
          consume_group<H, BITS>(st + i * GSPLIT * GBB, xlane0 + xo + i * GSPLIT * 128,
                                 xlane1 + xo + i * GSPLIT * 128, xslane + xso + i * GSPLIT * 64, lane,
                                 gq, yv);
      } else {
        for (int qd = rr; qd < cnt; qd += GSPLIT)
          consume_group<H, BITS>(st + (qd - rr) * GBB, xlane0 + xo + (uint32_t)(qd - rr) * 128u,
                                 xlane1 + xo + (uint32_t)(qd - rr) * 128u,
                                 xslane + xso + (uint32_t)(qd - rr) * 64u, lane, gq, yv);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[slot]);
    }
    if (++slot == (uint32_t)nst) {
      slot = 0;
      phase ^= 1u;
    }
    seg_hi = g + cnt;
    it.advance(cnt);
  }
  int last_b = -1;
  if (cur_b >= 0) {
    float z[ES];
    reduce(z);
    if (plan.cl) {
      cluster_finish(z, cur_b);
    } else if (seg_lo == 0 && seg_hi == G) {
      if (ok) store_share<H, ES>(y, y_f32, M, N, cur_b * BATCH + pr * TPW, rr, lane, z);
    } else {
      store_partial(z, first_seg);
      last_b = cur_b;
    }
  } else if (plan.cl) {  // (an empty range; not produced by make_plan) the cluster still meets twice
    cluster_sync_all();
    cluster_sync_all();
  }
  if (last_b >= 0) {
    named_barrier(1, CWARPS * 32);
    if (tid == 0) s_last2 = arrive(last_b);
    named_barrier(1, CWARPS * 32);
  }
  if (pend_b >= 0) {
    // the arrival warp's result for the first segment (made mid-range)
    if (!spin_wait(sm.seg1_arr, 0u, err)) ok = false;
    else if (s_last) merge(pend_b);
  }
  if (last_b >= 0 && s_last2) merge(last_b);
  if (TOPK) {
    // every consumer's logits are stored (CTA-scope order at the barrier);
    // the ring and the activation window are free
    __threadfence_block();
    named_barrier(1, CWARPS * 32);
    if (cta == 0 && tid == 0) {
      int *h = reinterpret_cast<int *>(topk.lists);
      h[0] = M;
      h[1] = plan.ctas;
      h[2] = topk.cap;
      h[3] = topk.k;
      h[4] = N;
    }
    const int c0 = (w0 / G) * BATCH * TILE_N, c1 = imin(N, (w1 / G) * BATCH * TILE_N);
    if (M >= 4)
      topk_lists<4>(static_cast<const float *>(y), M, N, c0, c1, topk, plan.ctas, cta, sm.ring, tid);
    else if (M >= 2)
      topk_lists<8>(static_cast<const float *>(y), M, N, c0, c1, topk, plan.ctas, cta, sm.ring, tid);
    else
      topk_lists<16>(static_cast<const float *>(y), M, N, c0, c1, topk, plan.ctas, cta, sm.ring, tid);
  }
}

}  // namespace qmm
}  // namespace sv

using namespace sv;

static size_t packed_bytes_bits(int N, int K, int group, int bits) {
  if (N < 1 || K < qmm::GROUP || K % qmm::GROUP != 0 || group != qmm::GROUP) return 0;
  const size_t NT = ((size_t)N + qmm::TILE_N - 1) / qmm::TILE_N;
  const size_t NB = (NT + qmm::BATCH - 1) / qmm::BATCH;
  return NB * (size_t)(K / qmm::GROUP) * (bits == 8 ? qmm::Pack<8>::GB : qmm::Pack<4>::GB);
}

static sv_status prepack_bits(const uint32_t *wq, const void *scales, const void *biases, int N, int K,
                              int group, int bits, void *packed_out, size_t packed_bytes,
                              sv_stream_t stream) {
  if (!wq || !scales || !biases || !packed_out) return SV_ERR_INVALID_ARG;
  if (N < 1 || K < 1 || group < 1) return SV_ERR_INVALID_ARG;
  if (group != qmm::GROUP || K % qmm::GROUP != 0) return SV_ERR_UNSUPPORTED;
  const size_t need = packed_bytes_bits(N, K, group, bits);
  if (packed_bytes < need) return SV_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(packed_out) % 16 != 0) return SV_ERR_INVALID_ARG;
  const int NT = (N + qmm::TILE_N - 1) / qmm::TILE_N, G = K / qmm::GROUP;
  const int NTP = (NT + qmm::BATCH - 1) / qmm::BATCH * qmm::BATCH;  // padded to whole batches
  const long long threads = (long long)NTP * G * 32;
  const int block = 256;
  const long long grid = (threads + block - 1) / block;
  if (grid > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
  cudaError_t e = launch(bits == 8 ? qmm::prepack8_kernel : qmm::prepack_kernel, dim3((unsigned)grid),
                         dim3(block), 0, reinterpret_cast<cudaStream_t>(stream), wq,
                         static_cast<const uint16_t *>(scales), static_cast<const uint16_t *>(biases),
                         N, K, NTP, G, static_cast<uint8_t *>(packed_out));
  return from_cuda(e);
}

static size_t workspace_bytes_bits(int M, int N, int K, int bits) {
  if (N < 1 || K < qmm::GROUP || K % qmm::GROUP != 0) return 0;
  const int sms = device_sm_count();
  if (sms <= 0) return 0;
  const int Mc = M < 1 ? 1 : (M > 16 ? 16 : M);
  const int H = Mc > 8 ? 2 : 1;
  return qmm::workspace_bytes(qmm::make_plan(N, K, H, Mc, sms, qmm::smem_optin(), bits));
}

// Launches a cluster plan if one pays for this shape and its clusters all
// fit on the device at once (at one CTA per SM a 152-SM GB300 runs 46
// clusters of 3, 36 of 4, 15 of 8), trying cluster sizes from 8 down; else
// the split plan if it pays; otherwise the stream-K plan `ps`.  The choice is
// cached per shape.
template <int H, int SG, int FM, int BITS>
static cudaError_t launch_qmm(const qmm::Plan &ps, int N, int K, int M, int sms, cudaStream_t s,
                              const __nv_bfloat16 *xp, const uint8_t *wp, void *y, int yf,
                              float *part, unsigned *counters, unsigned *err) {
  auto kern = qmm::qmm_kernel<H, SG, FM, BITS>;
  const qmm::TopkOut no_topk{nullptr, 0, 0};
  const size_t smem = qmm::smem_bytes(ps);
  const dim3 block(qmm::THREADS);
  static std::mutex mu;
  // (N, K, M, device) -> cluster size (>= 2), 1 for the split plan, 0 for stream-K
  static std::map<std::tuple<int, int, int, int>, int> chosen;
  int dev = 0;
  (void)cudaGetDevice(&dev);
  const auto key = std::make_tuple(N, K, M, dev);
  int cl = -1;
  {
    std::lock_guard<std::mutex> lk(mu);
    auto it = chosen.find(key);
    if (it != chosen.end()) cl = it->second;
  }
  if (cl < 0) {
    cl = 0;
    for (int c = 8; c >= 2; --c) {
      const qmm::Plan p = qmm::make_plan(N, K, H, M, sms, qmm::smem_optin(), BITS, c);
      if (!p.cl) break;
      if (p.cl < c) c = p.cl;  // (the shape caps the size)
      if (max_active_clusters(kern, qmm::THREADS, smem, p.cl) >= p.NB) {
        cl = p.cl;
        break;
      }
    }
    if (cl == 0 && qmm::make_plan(N, K, H, M, sms, qmm::smem_optin(), BITS, 0, true).sp) cl = 1;
    std::lock_guard<std::mutex> lk(mu);
    chosen[key] = cl;
  }
  if (cl >= 2) {
    const qmm::Plan pc = qmm::make_plan(N, K, H, M, sms, qmm::smem_optin(), BITS, cl);
    return launch_cluster(kern, dim3(pc.ctas), block, smem, s, pc.cl, xp, wp, y, yf, M, N, K, pc, part,
                          counters, err, no_topk);
  }
  // the stall test aid is not honoured under the cluster plan
  const int stall = (launch_flags() & SV_LAUNCH_TEST_STALL_COPY) ? 1 : 0;
  if (cl == 1) {
    qmm::Plan pt = qmm::make_plan(N, K, H, M, sms, qmm::smem_optin(), BITS, 0, true);
    pt.stall = stall;
    return launch(kern, dim3(pt.ctas), block, smem, s, xp, wp, y, yf, M, N, K, pt, part, counters, err,
                  no_topk);
  }
  qmm::Plan pk = ps;
  pk.stall = stall;
  return launch(kern, dim3(pk.ctas), block, smem, s, xp, wp, y, yf, M, N, K, pk, part, counters, err,
                no_topk);
}

static sv_status small_m_bits(const void *x_bf16, const void *packed_w, void *y, sv_dtype y_dtype,
                              int M, int N, int K, int group, int bits, void *workspace,
                              size_t ws_bytes, sv_stream_t stream) {
  if (!x_bf16 || !packed_w || !y) return SV_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || group < 1) return SV_ERR_INVALID_ARG;
  if (y_dtype != SV_BF16 && y_dtype != SV_F32) return SV_ERR_INVALID_ARG;
  if (M > 16 || group != qmm::GROUP || K % qmm::GROUP != 0) return SV_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(x_bf16) % 16 != 0 || reinterpret_cast<uintptr_t>(packed_w) % 16 != 0)
    return SV_ERR_INVALID_ARG;
  const int sms = device_sm_count();
  if (sms <= 0) return SV_ERR_CUDA;
  const int H = M > 8 ? 2 : 1;
  const qmm::Plan plan = qmm::make_plan(N, K, H, M, sms, qmm::smem_optin(), bits);
  const size_t need = qmm::workspace_bytes(plan);
  if (!workspace || ws_bytes < need) return SV_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return SV_ERR_INVALID_ARG;
  unsigned *err = device_error_word();
  if (!err) return SV_ERR_CUDA;
  unsigned *counters = static_cast<unsigned *>(workspace);
  float *part = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + qmm::counters_bytes(plan));
  const int yf = (y_dtype == SV_F32) ? 1 : 0;
  const auto *xp = static_cast<const __nv_bfloat16 *>(x_bf16);
  const auto *wp = static_cast<const uint8_t *>(packed_w);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
#define SV_QMM_LAUNCH(H_, SG_, FM_, B_) \
  launch_qmm<H_, SG_, FM_, B_>(plan, N, K, M, sms, s, xp, wp, y, yf, part, counters, err)
  if (bits == 8) {
    const int variant = (M <= 8 ? 0 : 2) + (plan.sg == 8 ? 0 : 1);
    switch (variant) {
      case 0: e = SV_QMM_LAUNCH(1, 8, 0, 8); break;
      case 1: e = SV_QMM_LAUNCH(1, 4, 0, 8); break;
      case 2: e = SV_QMM_LAUNCH(2, 8, 0, 8); break;
      default: e = SV_QMM_LAUNCH(2, 4, 0, 8); break;
    }
    return from_cuda(e);
  }
  if ((launch_flags() & SV_LAUNCH_QMM_CUDA_CORES) && plan.sg == 16 && (M == 1 || M == 4)) {
    e = M == 1 ? SV_QMM_LAUNCH(1, 16, 1, 4) : SV_QMM_LAUNCH(1, 16, 4, 4);
    return from_cuda(e);
  }
  const int variant = (M <= 8 ? 0 : 3) + (plan.sg == 16 ? 0 : plan.sg == 12 ? 1 : 2);
  switch (variant) {
    case 0: e = SV_QMM_LAUNCH(1, 16, 0, 4); break;
    case 1: e = SV_QMM_LAUNCH(1, 12, 0, 4); break;
    case 2: e = SV_QMM_LAUNCH(1, 8, 0, 4); break;
    case 3: e = SV_QMM_LAUNCH(2, 16, 0, 4); break;
    case 4: e = SV_QMM_LAUNCH(2, 12, 0, 4); break;
    default: e = SV_QMM_LAUNCH(2, 8, 0, 4); break;
  }
#undef SV_QMM_LAUNCH
  return from_cuda(e);
}

// The lm_head with the top-k lists epilogue: the plan must hold whole batches
// per CTA, and the row groups' scratch must fit the ring.
struct TopkPlan {
  qmm::Plan plan;
  int cap;
  sv_status st;
};
static TopkPlan topk_plan(int M, int N, int K) {
  TopkPlan t{};
  const int sms = device_sm_count();
  if (sms <= 0) {
    t.st = SV_ERR_CUDA;
    return t;
  }
  const int H = M > 8 ? 2 : 1;
  t.plan = qmm::make_plan(N, K, H, M, sms, qmm::smem_optin(), 4);
  t.cap = (t.plan.NB + t.plan.ctas - 1) / t.plan.ctas * qmm::BATCH * qmm::TILE_N;
  const int groups = M >= 4 ? 4 : (M >= 2 ? 2 : 1);
  const size_t scratch = (size_t)groups * qmm::topk_scratch(t.cap);
  t.st = (t.plan.aligned && scratch <= (size_t)t.plan.nst * t.plan.stage_bytes) ? SV_OK
                                                                                 : SV_ERR_UNSUPPORTED;
  return t;
}

extern "C" {

size_t qmm_topk_lists_bytes(int M, int N, int K) {
  if (M < 1 || M > 16 || N < 1 || K < qmm::GROUP || K % qmm::GROUP != 0) return 0;
  const TopkPlan t = topk_plan(M, N, K);
  if (t.st != SV_OK) return 0;
  return qmm::LISTS_HDR + (size_t)M * t.plan.ctas * qmm::list_stride(t.cap);
}

sv_status qmm_small_m_topk(const void *x_bf16, const void *packed_w, float *y, int M, int N, int K,
                           int group, sv_sampling_params params, void *lists, size_t lists_bytes,
                           void *workspace, size_t ws_bytes, sv_stream_t stream) {
  if (!x_bf16 || !packed_w || !y || !lists) return SV_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || group < 1) return SV_ERR_INVALID_ARG;
  const float T = params.temperature, tp = params.top_p;
  if (!(T >= 0.f) || !(T < INFINITY) || !(tp > 0.f && tp <= 1.f) || params.top_k < 0)
    return SV_ERR_INVALID_ARG;
  if (M > 16 || group != qmm::GROUP || K % qmm::GROUP != 0) return SV_ERR_UNSUPPORTED;
  // the candidate-list settings: temperature 0, or 0 < top_k <= 1024 below N
  const int k = T == 0.f ? 1 : params.top_k;
  if (T > 0.f && !(params.top_k > 0 && params.top_k <= 1024 && params.top_k < N))
    return SV_ERR_UNSUPPORTED;
  for (const void *p : {x_bf16, packed_w, (const void *)y, (const void *)lists})
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return SV_ERR_INVALID_ARG;
  const TopkPlan t = topk_plan(M, N, K);
  if (t.st != SV_OK) return t.st;
  const qmm::Plan &plan = t.plan;
  if (lists_bytes < qmm::LISTS_HDR + (size_t)M * plan.ctas * qmm::list_stride(t.cap))
    return SV_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < qmm::workspace_bytes(plan)) return SV_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return SV_ERR_INVALID_ARG;
  unsigned *err = device_error_word();
  if (!err) return SV_ERR_CUDA;
  unsigned *counters = static_cast<unsigned *>(workspace);
  float *part = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + qmm::counters_bytes(plan));
  const auto *xp = static_cast<const __nv_bfloat16 *>(x_bf16);
  const auto *wp = static_cast<const uint8_t *>(packed_w);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const dim3 grid(plan.ctas), block(qmm::THREADS);
  const size_t smem = qmm::smem_bytes(plan);
  const qmm::TopkOut to{static_cast<uint8_t *>(lists), k, t.cap};
  cudaError_t e;
#define SV_QMM_TOPK(H_, SG_)                                                                          \
  launch(qmm::qmm_kernel<H_, SG_, 0, 4, 1>, grid, block, smem, s, xp, wp, (void *)y, 1, M, N, K, plan, \
         part, counters, err, to)
  const int variant = (M <= 8 ? 0 : 3) + (plan.sg == 16 ? 0 : plan.sg == 12 ? 1 : 2);
  switch (variant) {
    case 0: e = SV_QMM_TOPK(1, 16); break;
    case 1: e = SV_QMM_TOPK(1, 12); break;
    case 2: e = SV_QMM_TOPK(1, 8); break;
    case 3: e = SV_QMM_TOPK(2, 16); break;
    case 4: e = SV_QMM_TOPK(2, 12); break;
    default: e = SV_QMM_TOPK(2, 8); break;
  }
#undef SV_QMM_TOPK
  return from_cuda(e);
}

size_t qmm_packed_bytes(int N, int K, int group) { return packed_bytes_bits(N, K, group, 4); }

sv_status qmm_prepack(const uint32_t *wq, const void *scales, const void *biases, int N, int K,
                      int group, void *packed_out, size_t packed_bytes, sv_stream_t stream) {
  return prepack_bits(wq, scales, biases, N, K, group, 4, packed_out, packed_bytes, stream);
}

size_t qmm_workspace_bytes(int M, int N, int K) { return workspace_bytes_bits(M, N, K, 4); }

sv_status qmm_small_m(const void *x_bf16, const void *packed_w, void *y, sv_dtype y_dtype, int M,
                      int N, int K, int group, void *workspace, size_t ws_bytes,
                      sv_stream_t stream) {
  return small_m_bits(x_bf16, packed_w, y, y_dtype, M, N, K, group, 4, workspace, ws_bytes, stream);
}

size_t qmm8_packed_bytes(int N, int K, int group) { return packed_bytes_bits(N, K, group, 8); }

sv_status qmm8_prepack(const uint32_t *wq, const void *scales, const void *biases, int N, int K,
                       int group, void *packed_out, size_t packed_bytes, sv_stream_t stream) {
  return prepack_bits(wq, scales, biases, N, K, group, 8, packed_out, packed_bytes, stream);
}

size_t qmm8_workspace_bytes(int M, int N, int K) { return workspace_bytes_bits(M, N, K, 8); }

sv_status qmm8_small_m(const void *x_bf16, const void *packed_w, void *y, sv_dtype y_dtype, int M,
                       int N, int K, int group, void *workspace, size_t ws_bytes,
                       sv_stream_t stream) {
  return small_m_bits(x_bf16, packed_w, y, y_dtype, M, N, K, group, 8, workspace, ws_bytes, stream);
}

}  // extern "C"
