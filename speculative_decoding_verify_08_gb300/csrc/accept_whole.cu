// accept_whole.cu -- spec_accept over the whole vocabulary: temperature > 0
// with top-k off, top-k >= V, or top-k beyond the candidate lists of
// accept.cu (more than 1024).
//
// Rule ("The fastest way to run local LLMs on a Mac", section "Why exact
// acceptance matters"; "Speculative decoding and MTP on Apple silicon",
// Facts): accept draft x iff u * q(x) < p(x); on the first rejection emit a
// sample of (p - q)+ and stop; if every draft is accepted emit a sample of
// the last target row.  p and q are truncated identically: temperature, then
// top-k (ties with the k-th logit kept), then top-p (a token is kept while
// the mass of strictly more likely kept tokens is below top_p).
//
// Representation.  For a row with largest logit zmax, token j has
//   x_j = (zmax - z_j) * log2(e) / T      and      E_j = round(2^62 * 2^-x_j),
// i.e. exp(z_j/T - zmax/T) as an integer with 62 fractional bits.  The
// truncated distribution is p_j = E_j / S over the kept tokens (key_j >= tau,
// keys being the order-preserving integer image of the logits), with S the
// sum of the kept E_j.  Every sum of E -- the normaliser, the masses walked
// by top-p, the kept mass, the inverse CDF's running sums -- is an exact
// integer sum, so results do not depend on the order of summation, the split
// over CTAs or atomics.  2^-x is evaluated in float-float arithmetic
// (Dekker's error-free products and sums) by a table-driven method (Tang,
// ACM TOMS 15(2), 1989: x = n + i/128 + r, 2^(-i/128) from a table, and
// exp(-r ln 2) by its Taylor polynomial to degree 5), relative error about
// 3e-14: the fp32 pipes carry the vocabulary-wide work, which on this part
// runs about 100x faster than fp64.
//
// Passes (V > 4096; rows = R * (2K+1), C CTAs per row):
//   max        row maximum (integer atomics on the key)
//   count      [top-k] bucket counts of x; the bucket where the count of
//              larger logits reaches k
//   compact    [top-k] that bucket's tokens into a list
//   select     [top-k] sort the list: the k-th largest key, tau_k
//   sum        Z = sum of E over the top-k set; [top-p] bucket counts of the
//              top-k set, from which bounds on the mass above each bucket give
//              the band of buckets that must hold the top-p boundary
//   compact    [top-p] the band's tokens into a list; exact mass above it
//   select     [top-p] sort the list, walk its tie groups with exact masses:
//              tau and S
//   decide     per round: the accept test of every draft, the first rejection
//   icdf       per round: one inverse-CDF sample of (p - q)+ or of the bonus
//              row, by exact chunk sums then a scan of one chunk
// A band (or a top-k bucket) longer than the list is narrowed by the select
// kernel itself over key ranges with exact counts and masses.  Rows of at most
// 4096 tokens take one select CTA per row for max, top-k, Z and top-p.
#include "accept_common.cuh"
#include "exp2_table.cuh"

namespace sv {
namespace whole {

using acc::fkey;
using acc::keyf;
using acc::load_logit;
using acc::load_logit_keep;
using acc::row_ptr;
typedef unsigned __int128 u128;

constexpr int THREADS = 256;      // multi-CTA passes, the inverse CDF
constexpr int SEL_THREADS = 512;  // one CTA per row: sort, scan, refinement
constexpr int NB = 8192;          // buckets of x; bucket b holds x within 1/256 of b/128
constexpr float RES = 128.f;      // buckets per unit of x (x < 64; the last bucket takes the rest)
constexpr int CAP = 4096;         // list entries one select CTA sorts
constexpr int SUB = 2048;         // sub-ranges per refinement level
constexpr float SLACK = 1e-4f;    // relative slack of the band's mass bounds (fp32 sums)
constexpr int MAX_LEVELS = 8;     // a 2^32-key range is one key after 3 levels

enum { MODE_SMALL = 0, MODE_TOPK = 1, MODE_TOPP = 2 };
enum { SUM_ONLY = 0, SUM_HIST = 1, COUNT_HIST = 2 };

// Per-row state (128 bytes).  Fields accumulated with atomics start at zero
// and are put back to zero by the pass that consumes them last.
struct Hdr {
  unsigned maxkey;      // key of the largest logit (reset by icdf)
  unsigned tau_k;       // kept by top-k iff key >= tau_k (top-k on)
  unsigned tau;         // kept iff key >= tau (top-p on)
  unsigned list_n;      // band entries appended (may exceed CAP; reset by select)
  unsigned band_lo;     // band of buckets holding the boundary
  unsigned band_hi;
  unsigned klo_inv;     // ~(smallest band key) (atomicMax; reset by select)
  unsigned khi;         // largest band key (atomicMax; reset by select)
  unsigned arrive;      // last-arriver counter of the histogram passes
  unsigned cnt_above;   // top-k: tokens in buckets before the band
  unsigned pad0, pad1;
  uint64_t z_lo, z_hi;  // Z = z_hi * 2^32 + z_lo (reset by icdf)
  uint64_t a_lo, a_hi;  // mass above the band, same split (reset by select)
  uint64_t s_lo, s_hi;  // kept mass S (top-p on), plain 128-bit value
};
static_assert(sizeof(Hdr) == 96, "header layout");
constexpr size_t HDR_BYTES = 128;

struct Job {
  int prow, qrow;  // rows of p and q (qrow < 0: sample p itself)
  int pos;         // output position of the sample
  float u;         // its uniform
};

struct Params {
  const void *tgt, *drf;
  const int32_t *drafts;
  const float *u;
  int32_t *out_tok, *out_n;
  int R, K, V, C, C2;
  float ch, cl;  // log2(e) / T as float-float
  int top_k;     // 0 = off
  float top_p;   // 1 = off
  uint8_t *hdr;  // [rows] HDR_BYTES
  unsigned *hist;     // [rows][NB] (V > CAP)
  uint64_t *list;     // [rows][CAP] (V > CAP)
  Job *jobs;          // [R]
  unsigned *icnt;     // [R]
  uint64_t *ipart;    // [R][C2][2]
};

__device__ __forceinline__ Hdr &hdr_of(const Params &p, long long row) {
  return *reinterpret_cast<Hdr *>(p.hdr + (size_t)row * HDR_BYTES);
}

// ------------------------------------------------------------- numerics --
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
// |a| >= |b|
__device__ __forceinline__ void fast_two_sum(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  e = __fsub_rn(b, __fsub_rn(s, a));
}

// x = (zmax - z) * c as an unevaluated float-float xh + xl (zmax >= z).
__device__ __forceinline__ void x_of(float zmax, float z, float ch, float cl, float &xh, float &xl) {
  float dh, dl;
  two_sum(zmax, -z, dh, dl);  // zmax - z exactly
  xh = __fmul_rn(dh, ch);
  const float xe = __fmaf_rn(dh, ch, -xh);  // exact error of dh * ch
  xl = __fmaf_rn(dh, cl, __fmaf_rn(dl, ch, xe));
}

// Bucket of x: the nearest integer to 128 x (as in efix), at most NB - 1;
// bucket b < NB - 1 holds x within 1/256 of b/128.  Monotone in x.
__device__ __forceinline__ int bucket_of(float xh) {
  const uint32_t j = __float_as_uint(__fadd_rn(__fmul_rn(xh, RES), 8388608.f)) - 0x4B000000u;
  return (int)min(j, (uint32_t)(NB - 1));
}

// round(2^62 * 2^-(xh + xl)) for xh >= 0; tab = EXP2_TAB in shared memory.
// x = n + i/128 + r with j = 128 n + i the nearest integer to 128 xh (found by
// adding 2^23, which rounds in the fp32 adder: no conversion instructions),
// |r| <= 1/256 + |xl|.
__device__ __forceinline__ uint64_t efix(float xh, float xl, const float2 *tab) {
  if (!(xh < 64.f)) return 0ull;  // below 2^-64 (or infinite)
  const float y = __fmul_rn(xh, 128.f);                          // exact
  const float t = __fadd_rn(y, 8388608.f);                       // 2^23 + round(y)
  const uint32_t j = __float_as_uint(t) - 0x4B000000u;           // round(y), 0..8192
  const float ry = __fsub_rn(y, __fsub_rn(t, 8388608.f));        // y - j, exact, |.| <= 1/2
  const int n = (int)(j >> 7), i = (int)(j & 127u);
  const float rh = __fmul_rn(ry, 0.0078125f);                    // exact
  // s = (rh + xl) * ln 2, float-float
  const float sh = __fmul_rn(rh, LN2_HI);
  const float se = __fmaf_rn(rh, LN2_HI, -sh);
  const float sl = __fmaf_rn(rh, LN2_LO, __fmaf_rn(xl, LN2_HI, se));
  // exp(-s) = 1 - s + s^2/2 - s^3/6 + s^4/24 - s^5/120   (|s| < 0.0028)
  const float s2h = __fmul_rn(sh, sh);
  const float s2l = __fmaf_rn(__fmul_rn(2.f, sh), sl, __fmaf_rn(sh, sh, -s2h));
  const float s3 = __fmul_rn(s2h, sh);
  const float tail = __fmul_rn(s3, __fmaf_rn(sh, __fmaf_rn(sh, -1.f / 120.f, 1.f / 24.f), -1.f / 6.f));
  float ah, ae, bh, be;
  fast_two_sum(1.f, -sh, ah, ae);
  fast_two_sum(ah, __fmul_rn(0.5f, s2h), bh, be);
  const float low = __fadd_rn(__fadd_rn(__fadd_rn(ae, be), __fsub_rn(__fmul_rn(0.5f, s2l), sl)), tail);
  float ph, pl;
  fast_two_sum(bh, low, ph, pl);
  // times 2^(-i/128)
  const float2 tt = tab[i];
  const float mh = __fmul_rn(tt.x, ph);
  const float me = __fmaf_rn(tt.x, ph, -mh);
  const float ml = __fmaf_rn(tt.x, pl, __fmaf_rn(tt.y, ph, me));
  // to 62 fractional bits from the bit fields (integer shifts; float-to-
  // integer conversions are not on the fp32 pipes), then times 2^-n with
  // rounding.  mh is in [0.498, 1.003] (exponent field 125..127); |ml| is below
  // 2^-22, its bits under 2^-62 are dropped (truncation toward zero).
  const uint32_t ubh = __float_as_uint(mh);
  const uint64_t Fh = (uint64_t)((ubh & 0x7FFFFFu) | 0x800000u) << (((ubh >> 23) & 0xFFu) - 88u);
  const uint32_t ubl = __float_as_uint(ml);
  const int el = (int)((ubl >> 23) & 0xFFu);
  const int64_t ml_m = (int64_t)((ubl & 0x7FFFFFu) | 0x800000u);
  const int shl = el - 88;
  int64_t Fl = el == 0 ? 0 : (shl >= 0 ? (ml_m << shl) : (shl > -24 ? (ml_m >> -shl) : 0));
  if (ubl >> 31) Fl = -Fl;
  const uint64_t F = Fh + (uint64_t)Fl;
  return n == 0 ? F : (((F >> (n - 1)) + 1ull) >> 1);
}

__device__ __forceinline__ uint64_t efix_z(float zmax, float z, const Params &p, const float2 *tab) {
  float xh, xl;
  x_of(zmax, z, p.ch, p.cl, xh, xl);
  return efix(xh, xl, tab);
}

__device__ __forceinline__ double u128_to_d(u128 v) {
  return (double)(uint64_t)(v >> 64) * 0x1p64 + (double)(uint64_t)v;
}

// f as m * 2^-sh with an integer m < 2^24 (f finite, f >= 0).
__device__ __forceinline__ void float_parts(float f, uint32_t &m, int &sh) {
  const uint32_t b = __float_as_uint(f);
  int e = (int)((b >> 23) & 0xFF);
  m = b & 0x7FFFFFu;
  if (e == 0) e = 1;
  else m |= 0x800000u;
  sh = 150 - e;
}
// floor(u * W), u in [0, 1)
__device__ __forceinline__ u128 floor_mul(float u, u128 W) {
  uint32_t m;
  int sh;
  float_parts(u, m, sh);
  const u128 prod = (u128)m * W;
  if (sh <= 0) return W;  // u >= 2^23: never for u < 1
  if (sh >= 128) return 0;
  return prod >> sh;
}
// ceil(f * Z), 0 < f <= 1
__device__ __forceinline__ u128 ceil_mul(float f, u128 Z) {
  uint32_t m;
  int sh;
  float_parts(f, m, sh);
  const u128 prod = (u128)m * Z;
  if (sh >= 128) return prod != 0 ? 1 : 0;
  return (prod + (((u128)1 << sh) - 1)) >> sh;
}

__device__ __forceinline__ void atomic_add_split(uint64_t *lo, uint64_t *hi, u128 v) {
  if (v == 0) return;
  atomicAdd(reinterpret_cast<unsigned long long *>(lo), (unsigned long long)(uint64_t)(v & 0xFFFFFFFFu));
  atomicAdd(reinterpret_cast<unsigned long long *>(hi), (unsigned long long)(uint64_t)(v >> 32));
}
__device__ __forceinline__ u128 read_split(const uint64_t *lo, const uint64_t *hi) {
  return ((u128)__ldcg(reinterpret_cast<const unsigned long long *>(hi)) << 32) +
         (u128)__ldcg(reinterpret_cast<const unsigned long long *>(lo));
}

// ---------------------------------------------------- block reductions --
__device__ __forceinline__ u128 shfl_xor_u128(u128 v, int m) {
  const uint64_t lo = __shfl_xor_sync(0xffffffffu, (unsigned long long)(uint64_t)v, m);
  const uint64_t hi = __shfl_xor_sync(0xffffffffu, (unsigned long long)(uint64_t)(v >> 64), m);
  return ((u128)hi << 64) | lo;
}
__device__ __forceinline__ u128 shfl_up_u128(u128 v, int d) {
  const uint64_t lo = __shfl_up_sync(0xffffffffu, (unsigned long long)(uint64_t)v, d);
  const uint64_t hi = __shfl_up_sync(0xffffffffu, (unsigned long long)(uint64_t)(v >> 64), d);
  return ((u128)hi << 64) | lo;
}

template <int NT>
__device__ u128 block_sum_u128(u128 v, u128 *sm) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += shfl_xor_u128(v, m);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = v;
  __syncthreads();
  u128 t = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) t += sm[w];
  return t;
}

// Exclusive prefix of v over the block (thread order); total in *total.
template <int NT>
__device__ u128 block_excl_u128(u128 v, u128 &total, u128 *sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  u128 inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const u128 o = shfl_up_u128(inc, d);
    if (lane >= d) inc += o;
  }
  __syncthreads();
  if (lane == 31) sm[warp] = inc;
  __syncthreads();
  u128 base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    if (w < warp) base += sm[w];
    tot += sm[w];
  }
  total = tot;
  return base + inc - v;
}

template <int NT, typename V>
__device__ V block_excl_scalar(V v, V &total, V *sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  V inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const V o = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += o;
  }
  __syncthreads();
  if (lane == 31) sm[warp] = inc;
  __syncthreads();
  V base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    if (w < warp) base += sm[w];
    tot += sm[w];
  }
  total = tot;
  return base + inc - v;
}

template <int NT>
__device__ int block_max_int(int v, int *sm) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, m));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = v;
  __syncthreads();
  int t = sm[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) t = max(t, sm[w]);
  return t;
}
template <int NT>
__device__ unsigned block_max_u32(unsigned v, unsigned *sm) {
  v = __reduce_max_sync(0xffffffffu, v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned t = sm[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) t = max(t, sm[w]);
  return t;
}

__device__ __forceinline__ void load_table(float2 *tab) {
  for (int i = threadIdx.x; i < 128; i += blockDim.x) tab[i] = EXP2_TAB[i];
}

// Last CTA of a group of `n` to arrive on *ctr (acquire-release; the counter
// is put back to zero).  Call with the whole block after its global writes.
__device__ __forceinline__ bool last_arriver(unsigned *ctr, unsigned n, int *s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    unsigned prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(ctr) : "memory");
    *s_flag = prev == n - 1;
    if (*s_flag) *ctr = 0u;
  }
  __syncthreads();
  return *s_flag != 0;
}

// Bitonic sort of a[0..P2) in descending order (P2 a power of two).
template <int NT>
__device__ void sort_desc(uint64_t *a, int P2) {
  for (int size = 2; size <= P2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int t = threadIdx.x; t < P2 / 2; t += NT) {
        const int i = 2 * t - (t & (stride - 1));  // i has bit `stride` clear
        const int q = i + stride;
        const bool desc = (i & size) == 0;
        const uint64_t x = a[i], y = a[q];
        if ((x < y) == desc) {
          a[i] = y;
          a[q] = x;
        }
      }
      __syncthreads();
    }
  }
}

__device__ __forceinline__ int pow2_at_least(int n) {
  int p = 1;
  while (p < n) p <<= 1;
  return p;
}

// Sorted-list entry: key in the high word, ~index in the low word, so that a
// descending sort orders by key descending, then index ascending.
__device__ __forceinline__ uint64_t entry(uint32_t key, uint32_t idx) {
  return ((uint64_t)key << 32) | (uint32_t)~idx;
}
__device__ __forceinline__ uint32_t entry_key(uint64_t e) { return (uint32_t)(e >> 32); }

// ------------------------------------------------------------------ max --
template <typename T>
__global__ void __launch_bounds__(THREADS) max_kernel(const Params p) {
  __shared__ unsigned s_red[THREADS / 32];
  pdl_wait();
  const int rows2 = 2 * p.K + 1;
  const long long row = blockIdx.x / p.C;
  const int chunk = blockIdx.x % p.C;
  const T *z = row_ptr(static_cast<const T *>(p.tgt), static_cast<const T *>(p.drf),
                       (int)(row / rows2), (int)(row % rows2), p.K, p.V);
  const long long lo = (long long)chunk * p.V / p.C, hi = (long long)(chunk + 1) * p.V / p.C;
  unsigned m = 0;
  for (long long i = lo + threadIdx.x; i < hi; i += THREADS) m = max(m, fkey(load_logit_keep(z, i)));
  m = block_max_u32<THREADS>(m, s_red);
  if (threadIdx.x == 0) atomicMax(&hdr_of(p, row).maxkey, m);
}

// ------------------------------------------------------- band searches --
// Counts of the row's buckets in cnt[NB] (shared).  The bucket where the
// number of larger-logit tokens reaches k.
__device__ void band_by_count(const Params &p, Hdr &h, const unsigned *cnt, unsigned *s_u, int *s_i) {
  constexpr int PER = NB / THREADS;
  const int b0 = threadIdx.x * PER;
  unsigned loc = 0;
  for (int e = 0; e < PER; ++e) loc += cnt[b0 + e];
  unsigned tot;
  unsigned cum = block_excl_scalar<THREADS, unsigned>(loc, tot, s_u);
  int found = -1;
  unsigned above = 0;
  for (int e = 0; e < PER; ++e) {
    const unsigned c = cnt[b0 + e];
    if (found < 0 && c > 0 && cum < (unsigned)p.top_k && (unsigned)p.top_k <= cum + c) {
      found = b0 + e;
      above = cum;
    }
    cum += c;
  }
  if (found >= 0) {  // exactly one thread
    h.band_lo = (unsigned)found;
    h.band_hi = (unsigned)found;
    h.cnt_above = above;
  }
}

// Counts of the top-k set's buckets in cnt[NB]; Z in units of 2^-62.  Bounds
// on the mass above each bucket (every token of bucket b weighs between
// 2^-(b+1/2)/128 and 2^-(b-1/2)/128 of the largest) give the band of buckets
// that holds the last kept tie group of top-p.
__device__ void band_by_mass(const Params &p, Hdr &h, const unsigned *cnt, u128 Z, float *s_f,
                             int *s_i) {
  constexpr int PER = NB / THREADS;
  const int b0 = threadIdx.x * PER;
  const float thr = p.top_p * (float)(u128_to_d(Z) * 0x1p-62);
  float su = 0.f, sl = 0.f;
  for (int e = 0; e < PER; ++e) {
    const int b = b0 + e;
    const float c = (float)cnt[b];
    su += c * (b == 0 ? 1.f : exp2f(-((float)b - 0.5f) / RES));
    sl += (b == NB - 1) ? 0.f : c * exp2f(-((float)b + 0.5f) / RES);
  }
  float tu, tl;
  float U = block_excl_scalar<THREADS, float>(su, tu, s_f);
  float L = block_excl_scalar<THREADS, float>(sl, tl, s_f);
  int mylo = 0x7fffffff, myhi = -1, mylast = -1;
  for (int e = 0; e < PER; ++e) {
    const int b = b0 + e;
    const unsigned c = cnt[b];
    const float wu = (float)c * (b == 0 ? 1.f : exp2f(-((float)b - 0.5f) / RES));
    const float wl = (b == NB - 1) ? 0.f : (float)c * exp2f(-((float)b + 0.5f) / RES);
    if (c) {
      if (mylo == 0x7fffffff && (U + wu) * (1.f + SLACK) >= thr) mylo = b;
      if (L * (1.f - SLACK) < thr) myhi = b;
      mylast = b;
    }
    U += wu;
    L += wl;
  }
  const int lo = -block_max_int<THREADS>(-mylo, s_i);
  const int hi = block_max_int<THREADS>(myhi, s_i);
  const int last = block_max_int<THREADS>(mylast, s_i);
  if (threadIdx.x == 0) {
    int blo = lo == 0x7fffffff ? last : lo;
    int bhi = hi < 0 ? last : hi;
    if (blo > bhi) {
      const int t = blo;
      blo = bhi;
      bhi = t;
    }
    h.band_lo = (unsigned)blo;
    h.band_hi = (unsigned)bhi;
  }
}

// ------------------------------------------------------------------ sum --
// SUM_ONLY: Z.  SUM_HIST: Z and the top-k set's bucket counts, then (last
// CTA of the row) the top-p band.  COUNT_HIST: bucket counts of every token,
// then the top-k bucket.
template <typename T, int MODE>
__global__ void __launch_bounds__(THREADS) sum_kernel(const Params p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  unsigned *cnt = reinterpret_cast<unsigned *>(smem_raw);  // [NB] (histogram modes)
  __shared__ float2 tab[128];
  __shared__ u128 s_u128[THREADS / 32];
  __shared__ float s_f[THREADS / 32];
  __shared__ unsigned s_u[THREADS / 32];
  __shared__ int s_i[THREADS / 32];
  __shared__ int s_last;
  pdl_wait();
  const int rows2 = 2 * p.K + 1;
  const long long row = blockIdx.x / p.C;
  const int chunk = blockIdx.x % p.C;
  Hdr &h = hdr_of(p, row);
  const T *z = row_ptr(static_cast<const T *>(p.tgt), static_cast<const T *>(p.drf),
                       (int)(row / rows2), (int)(row % rows2), p.K, p.V);
  const long long lo = (long long)chunk * p.V / p.C, hi = (long long)(chunk + 1) * p.V / p.C;
  const float zmax = keyf(h.maxkey);
  const unsigned tk = (MODE != COUNT_HIST && p.top_k > 0) ? h.tau_k : 0u;
  load_table(tab);
  if (MODE != SUM_ONLY)
    for (int b = threadIdx.x; b < NB; b += THREADS) cnt[b] = 0u;
  __syncthreads();
  u128 acc = 0;
  for (long long i = lo + threadIdx.x; i < hi; i += THREADS) {
    const float zi = load_logit_keep(z, i);
    if (fkey(zi) < tk) continue;
    float xh, xl;
    x_of(zmax, zi, p.ch, p.cl, xh, xl);
    if (MODE != COUNT_HIST) acc += efix(xh, xl, tab);
    if (MODE != SUM_ONLY) atomicAdd(&cnt[bucket_of(xh)], 1u);
  }
  if (MODE != COUNT_HIST) {
    acc = block_sum_u128<THREADS>(acc, s_u128);
    if (threadIdx.x == 0) atomic_add_split(&h.z_lo, &h.z_hi, acc);
  }
  if (MODE == SUM_ONLY) return;
  __syncthreads();
  unsigned *gh = p.hist + (size_t)row * NB;
  for (int b = threadIdx.x; b < NB; b += THREADS)
    if (cnt[b]) atomicAdd(&gh[b], cnt[b]);
  if (!last_arriver(&h.arrive, (unsigned)p.C, &s_last)) return;
  for (int b = threadIdx.x; b < NB; b += THREADS) {
    cnt[b] = __ldcg(&gh[b]);
    gh[b] = 0u;  // ready for the next pass or call
  }
  __syncthreads();
  if (MODE == COUNT_HIST) band_by_count(p, h, cnt, s_u, s_i);
  else band_by_mass(p, h, cnt, read_split(&h.z_lo, &h.z_hi), s_f, s_i);
}

// -------------------------------------------------------------- compact --
// The band's tokens into the row's list (key, index); their least and
// largest keys; [top-p] the exact mass of the top-k set above the band.
template <typename T, int MODE>
__global__ void __launch_bounds__(THREADS) compact_kernel(const Params p) {
  __shared__ float2 tab[128];
  __shared__ u128 s_u128[THREADS / 32];
  __shared__ unsigned s_u[THREADS / 32];
  pdl_wait();
  const int rows2 = 2 * p.K + 1;
  const long long row = blockIdx.x / p.C;
  const int chunk = blockIdx.x % p.C;
  Hdr &h = hdr_of(p, row);
  const T *z = row_ptr(static_cast<const T *>(p.tgt), static_cast<const T *>(p.drf),
                       (int)(row / rows2), (int)(row % rows2), p.K, p.V);
  const long long lo = (long long)chunk * p.V / p.C, hi = (long long)(chunk + 1) * p.V / p.C;
  const float zmax = keyf(h.maxkey);
  const unsigned tk = (MODE == MODE_TOPP && p.top_k > 0) ? h.tau_k : 0u;
  const int blo = (int)h.band_lo, bhi = (int)h.band_hi;
  uint64_t *list = p.list + (size_t)row * CAP;
  if (MODE == MODE_TOPP) {
    load_table(tab);
    __syncthreads();
  }
  const int lane = threadIdx.x & 31;
  u128 acc = 0;
  unsigned kmin_inv = 0, kmax = 0;
  for (long long base = lo; base < hi; base += THREADS) {
    const long long i = base + threadIdx.x;
    bool in = false;
    uint32_t key = 0;
    if (i < hi) {
      const float zi = load_logit_keep(z, i);
      key = fkey(zi);
      if (key >= tk) {
        float xh, xl;
        x_of(zmax, zi, p.ch, p.cl, xh, xl);
        const int b = bucket_of(xh);
        in = b >= blo && b <= bhi;
        if (MODE == MODE_TOPP && b < blo) acc += efix(xh, xl, tab);
      }
    }
    const unsigned m = __ballot_sync(0xffffffffu, in);
    if (m) {
      const int leader = __ffs(m) - 1;
      unsigned pos = 0;
      if (lane == leader) pos = atomicAdd(&h.list_n, (unsigned)__popc(m));
      pos = __shfl_sync(0xffffffffu, pos, leader) + __popc(m & ((1u << lane) - 1u));
      if (in) {
        if (pos < (unsigned)CAP) list[pos] = entry(key, (uint32_t)i);
        kmin_inv = max(kmin_inv, ~key);
        kmax = max(kmax, key);
      }
    }
  }
  kmin_inv = block_max_u32<THREADS>(kmin_inv, s_u);
  kmax = block_max_u32<THREADS>(kmax, s_u);
  if (threadIdx.x == 0 && kmax != 0u) {
    atomicMax(&h.klo_inv, kmin_inv);
    atomicMax(&h.khi, kmax);
  }
  if (MODE == MODE_TOPP) {
    acc = block_sum_u128<THREADS>(acc, s_u128);
    if (threadIdx.x == 0) atomic_add_split(&h.a_lo, &h.a_hi, acc);
  }
}

// --------------------------------------------------------------- select --
struct SelSmem {
  uint64_t *a;  // sorted entries [cap]
  uint64_t *e;  // E of each entry [cap] (top-p); aliased by the refinement's masses
  unsigned *c;  // refinement counts [SUB]
};

// Exact walk of a sorted list a[0..n) (descending keys) with E in e[]: the
// last tie group whose mass above (above0 plus the list's entries before it)
// is below TH.  Writes *tau and *S (kept mass: above0 + the list up to the
// end of that group).
__device__ void walk_groups(const uint64_t *a, const uint64_t *e, int n, u128 above0, u128 TH,
                            unsigned *tau, u128 *S, u128 *s_u128, int *s_i, u128 *s_S) {
  constexpr int NT = SEL_THREADS;
  const int per = (n + NT - 1) / NT;
  const int t0 = min(n, (int)threadIdx.x * per), t1 = min(n, t0 + per);
  u128 loc = 0;
  for (int i = t0; i < t1; ++i) loc += e[i];
  u128 tot;
  u128 cum = above0 + block_excl_u128<NT>(loc, tot, s_u128);
  int cand = -1;
  for (int i = t0; i < t1; ++i) {
    if ((i == 0 || entry_key(a[i]) != entry_key(a[i - 1])) && cum < TH) cand = i;
    cum += e[i];
  }
  int g = block_max_int<NT>(cand, s_i);
  if (g < 0) g = 0;  // unreachable: the band holds the boundary
  const uint32_t kg = entry_key(a[g]);
  cum = above0 + block_excl_u128<NT>(loc, tot, s_u128);
  for (int i = t0; i < t1; ++i) {
    cum += e[i];
    if (entry_key(a[i]) == kg && (i + 1 == n || entry_key(a[i + 1]) != kg)) *s_S = cum;
  }
  __syncthreads();
  *tau = kg;
  *S = *s_S;
}

// One refinement level over the row: counts (and masses) of keys in
// [klo, khi] per sub-range of SUB; returns the crossing sub-range's key
// range, its count, and updates need (top-k) or above (top-p).
template <typename T, int MODE>
__device__ void refine(const Params &p, const T *z, float zmax, const float2 *tab, SelSmem &sm,
                       uint32_t &klo, uint32_t &khi, unsigned &need, u128 &above, u128 TH,
                       unsigned &cnt_out, u128 &mass_out, unsigned *s_u, u128 *s_u128, int *s_i) {
  constexpr int NT = SEL_THREADS;
  uint64_t *mlo = sm.e, *mhi = sm.e + SUB;
  const uint64_t nr = (uint64_t)khi - klo + 1;
  for (int b = threadIdx.x; b < SUB; b += NT) {
    sm.c[b] = 0u;
    if (MODE == MODE_TOPP) {
      mlo[b] = 0ull;
      mhi[b] = 0ull;
    }
  }
  __syncthreads();
  for (long long i = threadIdx.x; i < p.V; i += NT) {
    const float zi = load_logit_keep(z, i);
    const uint32_t key = fkey(zi);
    if (key < klo || key > khi) continue;
    const int sb = (int)(((uint64_t)(khi - key) * SUB) / nr);
    atomicAdd(&sm.c[sb], 1u);
    if (MODE == MODE_TOPP) {
      const uint64_t E = efix_z(zmax, zi, p, tab);
      atomicAdd(reinterpret_cast<unsigned long long *>(&mlo[sb]), (unsigned long long)(E & 0xFFFFFFFFull));
      atomicAdd(reinterpret_cast<unsigned long long *>(&mhi[sb]), (unsigned long long)(E >> 32));
    }
  }
  __syncthreads();
  constexpr int PER = SUB / NT;
  const int b0 = threadIdx.x * PER;
  int sb = -1;
  unsigned cntb = 0;
  u128 massb = 0;
  if (MODE == MODE_TOPK) {
    unsigned loc = 0;
    for (int e = 0; e < PER; ++e) loc += sm.c[b0 + e];
    unsigned tot;
    unsigned cum = block_excl_scalar<NT, unsigned>(loc, tot, s_u);
    int found = -1;
    for (int e = 0; e < PER; ++e) {
      const unsigned c = sm.c[b0 + e];
      if (found < 0 && c > 0 && cum < need && need <= cum + c) found = b0 + e;
      if (found < 0) cum += c;
    }
    // the crossing sub-range's thread publishes need
    sb = block_max_int<NT>(found, s_i);
    if (sb < 0) {  // unreachable: need is within the range's count
      sb = 0;
      if (threadIdx.x == 0) s_u[0] = need;
    } else if (found == sb) {
      s_u[0] = need - cum;
    }
    __syncthreads();
    need = s_u[0];
    cntb = sm.c[sb];
    __syncthreads();
  } else {
    u128 loc = 0;
    for (int e = 0; e < PER; ++e) loc += ((u128)mhi[b0 + e] << 32) + mlo[b0 + e];
    u128 tot;
    u128 cum = above + block_excl_u128<NT>(loc, tot, s_u128);
    int found = -1;
    u128 cum_at = 0;
    for (int e = 0; e < PER; ++e) {
      const int b = b0 + e;
      if (sm.c[b] > 0 && cum < TH) {
        found = b;
        cum_at = cum;
      }
      cum += ((u128)mhi[b] << 32) + mlo[b];
    }
    sb = block_max_int<NT>(found, s_i);
    if (sb < 0) {  // unreachable: the range holds the last kept group
      sb = 0;
      if (threadIdx.x == 0) s_u128[0] = above;
    } else if (found == sb) {
      s_u128[0] = cum_at;
    }
    __syncthreads();
    above = s_u128[0];
    cntb = sm.c[sb];
    massb = ((u128)mhi[sb] << 32) + mlo[sb];
    __syncthreads();
  }
  // key range of sub-range sb: (khi - key) * SUB / nr == sb
  const uint64_t d0 = ((uint64_t)sb * nr + SUB - 1) / SUB;
  const uint64_t d1 = ((uint64_t)(sb + 1) * nr + SUB - 1) / SUB - 1;
  const uint32_t nhi = khi - (uint32_t)d0, nlo = khi - (uint32_t)d1;
  klo = nlo;
  khi = nhi;
  cnt_out = cntb;
  mass_out = massb;
}

// One CTA per row.  MODE_SMALL (V <= CAP): the whole row.  MODE_TOPK: tau_k
// from the band list.  MODE_TOPP: tau and S from the band list.
template <typename T, int MODE>
__global__ void __launch_bounds__(SEL_THREADS) select_kernel(const Params p) {
  constexpr int NT = SEL_THREADS;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ float2 tab[128];
  __shared__ u128 s_u128[NT / 32];
  __shared__ unsigned s_u[NT / 32];
  __shared__ int s_i[NT / 32];
  __shared__ u128 s_S;
  __shared__ unsigned s_n;
  pdl_wait();
  const int rows2 = 2 * p.K + 1;
  const long long row = blockIdx.x;
  Hdr &h = hdr_of(p, row);
  const T *z = row_ptr(static_cast<const T *>(p.tgt), static_cast<const T *>(p.drf),
                       (int)(row / rows2), (int)(row % rows2), p.K, p.V);
  const int cap = MODE == MODE_SMALL ? pow2_at_least(p.V) : CAP;
  SelSmem sm;
  sm.a = reinterpret_cast<uint64_t *>(smem_raw);
  sm.e = sm.a + cap;
  sm.c = reinterpret_cast<unsigned *>(sm.e + (MODE == MODE_TOPP ? cap : 0));
  load_table(tab);

  if (MODE == MODE_SMALL) {
    const int V = p.V;
    unsigned mk = 0;
    for (int i = threadIdx.x; i < cap; i += NT) {
      uint64_t en = 0ull;
      if (i < V) {
        const uint32_t key = fkey(load_logit(z, i));
        en = entry(key, (uint32_t)i);
        mk = max(mk, key);
      }
      sm.a[i] = en;
    }
    mk = block_max_u32<NT>(mk, s_u);
    const float zmax = keyf(mk);
    const bool has_k = p.top_k > 0, has_p = p.top_p < 1.f;
    if (has_k || has_p) sort_desc<NT>(sm.a, cap);
    // the top-k set is a[0..m)
    unsigned tk = 0;
    int m = V;
    if (has_k) {
      tk = entry_key(sm.a[p.top_k - 1]);
      int first_below = V;
      for (int i = threadIdx.x; i < V; i += NT)
        if (entry_key(sm.a[i]) < tk && (i == 0 || entry_key(sm.a[i - 1]) >= tk)) first_below = i;
      m = -block_max_int<NT>(-first_below, s_i);
    }
    u128 loc = 0;
    for (int i = threadIdx.x; i < m; i += NT) {
      const uint64_t E = efix_z(zmax, keyf(entry_key(sm.a[i])), p, tab);
      sm.e[i] = E;
      loc += E;
    }
    const u128 Z = block_sum_u128<NT>(loc, s_u128);
    unsigned tau = tk;
    u128 S = Z;
    if (has_p) walk_groups(sm.a, sm.e, m, 0, ceil_mul(p.top_p, Z), &tau, &S, s_u128, s_i, &s_S);
    if (threadIdx.x == 0) {
      h.maxkey = mk;
      h.tau_k = tk;
      h.tau = tau;
      h.z_lo = (uint64_t)(Z & 0xFFFFFFFFu);
      h.z_hi = (uint64_t)(Z >> 32);
      h.s_lo = (uint64_t)S;
      h.s_hi = (uint64_t)(S >> 64);
    }
    return;
  }

  // ---- band modes ----
  const float zmax = keyf(h.maxkey);
  const unsigned n = h.list_n;
  uint32_t klo = ~h.klo_inv, khi = h.khi;
  unsigned need = MODE == MODE_TOPK ? (unsigned)p.top_k - h.cnt_above : 0u;
  u128 above = MODE == MODE_TOPP ? read_split(&h.a_lo, &h.a_hi) : 0;
  const u128 Z = MODE == MODE_TOPP ? read_split(&h.z_lo, &h.z_hi) : 0;
  const u128 TH = MODE == MODE_TOPP ? ceil_mul(p.top_p, Z) : 0;
  const uint64_t *glist = p.list + (size_t)row * CAP;
  int nl = -1;           // entries in sm.a to finish from (-1: single key, no list)
  unsigned single = 0;   // the key when the boundary range is one key
  u128 single_mass = 0;
  if (n <= (unsigned)CAP) {
    for (int i = threadIdx.x; i < (int)n; i += NT) sm.a[i] = __ldcg(glist + i);
    nl = (int)n;
  } else {
    // the band outgrew the list: narrow the key range by exact counts and
    // masses, one level per pass over the row
    __syncthreads();
    for (int level = 0; level < MAX_LEVELS; ++level) {
      unsigned c;
      u128 mass;
      refine<T, MODE>(p, z, zmax, tab, sm, klo, khi, need, above, TH, c, mass, s_u, s_u128, s_i);
      if (klo == khi) {
        single = klo;
        single_mass = mass;
        break;
      }
      if (c <= (unsigned)CAP) {
        if (threadIdx.x == 0) s_n = 0u;
        __syncthreads();
        for (long long i = threadIdx.x; i < p.V; i += NT) {
          const uint32_t key = fkey(load_logit_keep(z, i));
          if (key >= klo && key <= khi) {
            const unsigned pos = atomicAdd(&s_n, 1u);
            if (pos < (unsigned)CAP) sm.a[pos] = entry(key, (uint32_t)i);
          }
        }
        __syncthreads();
        nl = (int)min(s_n, (unsigned)CAP);
        break;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {  // ready for the next call
    h.list_n = 0u;
    h.klo_inv = 0u;
    h.khi = 0u;
    h.a_lo = 0ull;
    h.a_hi = 0ull;
  }
  if (MODE == MODE_TOPK) {
    unsigned tk;
    if (nl < 0) {
      tk = single;
    } else {
      const int P2 = pow2_at_least(nl);
      for (int i = nl + threadIdx.x; i < P2; i += NT) sm.a[i] = 0ull;
      __syncthreads();
      sort_desc<NT>(sm.a, P2);
      tk = entry_key(sm.a[need - 1]);
    }
    if (threadIdx.x == 0) h.tau_k = tk;
  } else {
    unsigned tau;
    u128 S;
    if (nl < 0) {
      tau = single;
      S = above + single_mass;
    } else {
      const int P2 = pow2_at_least(nl);
      for (int i = nl + threadIdx.x; i < P2; i += NT) sm.a[i] = 0ull;
      __syncthreads();
      sort_desc<NT>(sm.a, P2);
      for (int i = threadIdx.x; i < nl; i += NT) sm.e[i] = efix_z(zmax, keyf(entry_key(sm.a[i])), p, tab);
      __syncthreads();
      walk_groups(sm.a, sm.e, nl, above, TH, &tau, &S, s_u128, s_i, &s_S);
    }
    if (threadIdx.x == 0) {
      h.tau = tau;
      h.s_lo = (uint64_t)S;
      h.s_hi = (uint64_t)(S >> 64);
    }
  }
}

// ---------------------------------------------------------- row access --
struct RowView {
  const void *z;
  float zmax;
  unsigned tau;
  u128 S;
};

template <typename T>
__device__ __forceinline__ RowView row_view(const Params &p, long long row) {
  const int rows2 = 2 * p.K + 1;
  const Hdr &h = hdr_of(p, row);
  RowView v;
  v.z = row_ptr(static_cast<const T *>(p.tgt), static_cast<const T *>(p.drf), (int)(row / rows2),
                (int)(row % rows2), p.K, p.V);
  v.zmax = keyf(h.maxkey);
  const bool has_p = p.top_p < 1.f, has_k = p.top_k > 0;
  v.tau = has_p ? h.tau : (has_k ? h.tau_k : 0u);
  v.S = has_p ? (((u128)h.s_hi << 64) | h.s_lo) : (((u128)h.z_hi << 32) + h.z_lo);
  return v;
}

// E_x of a kept token, 0 otherwise.
template <typename T>
__device__ __forceinline__ uint64_t kept_E(const Params &p, const RowView &v, long long x,
                                           const float2 *tab) {
  const float zx = load_logit_keep(static_cast<const T *>(v.z), x);
  if (fkey(zx) < v.tau) return 0ull;
  return efix_z(v.zmax, zx, p, tab);
}

// --------------------------------------------------------------- decide --
// One warp per round: every draft's accept test, the first rejection, the
// accepted tokens, and the inverse-CDF job of the round's final sample.
template <typename T>
__global__ void __launch_bounds__(32) decide_kernel(const Params p) {
  __shared__ float2 tab[128];
  pdl_wait();
  load_table(tab);
  __syncwarp();
  const int r = blockIdx.x, lane = threadIdx.x, K = p.K;
  const long long base = (long long)r * (2 * K + 1);
  bool acc = true;
  int x = -1;
  if (lane < K) {
    x = p.drafts[(size_t)r * K + lane];
    // u q(x) < p(x) with p(x) = Ep/Sp, q(x) = Eq/Sq, without divisions:
    // u Eq Sp < Ep Sq (a token outside both supports is rejected)
    double lhs = 0.0, rhs = 0.0;
    if (x >= 0 && x < p.V) {
      const RowView vp = row_view<T>(p, base + lane), vq = row_view<T>(p, base + K + 1 + lane);
      const double Ep = (double)kept_E<T>(p, vp, x, tab), Eq = (double)kept_E<T>(p, vq, x, tab);
      lhs = (double)p.u[(size_t)r * (K + 1) + lane] * Eq * u128_to_d(vp.S);
      rhs = Ep * u128_to_d(vq.S);
    }
    acc = lhs < rhs;
  }
  const unsigned rej = __ballot_sync(0xffffffffu, lane < K && !acc);
  const int n = rej ? __ffs(rej) - 1 : K;
  int32_t *tok = p.out_tok + (size_t)r * (K + 1);
  if (lane < n) tok[lane] = x;
  for (int i = n + 1 + lane; i <= K; i += 32) tok[i] = -1;
  if (lane == 0) {
    p.out_n[r] = n;
    Job j;
    j.prow = (int)(n < K ? base + n : base + K);
    j.qrow = n < K ? (int)(base + K + 1 + n) : -1;
    j.pos = n;
    j.u = p.u[(size_t)r * (K + 1) + K];
    p.jobs[r] = j;
  }
}

// ----------------------------------------------------------------- icdf --
struct Weights {
  RowView vp, vq;
  bool resid;
  uint64_t ap, aq;  // 2^124 / S (residual)
};

template <typename T>
__device__ __forceinline__ uint64_t weight(const Params &p, const Weights &w, long long i,
                                           const float2 *tab) {
  const uint64_t Ep = kept_E<T>(p, w.vp, i, tab);
  if (!w.resid) return Ep;
  const uint64_t Eq = kept_E<T>(p, w.vq, i, tab);
  // (p_i - q_i)+ * 2^62 = (Ep/Sp - Eq/Sq)+ * 2^62
  const u128 a = (u128)Ep * w.ap, b = (u128)Eq * w.aq;
  return a > b ? (uint64_t)((a - b) >> 62) : 0ull;
}

// The first index of [lo, hi) whose running weight sum exceeds t (t below the
// range's total), by contiguous per-thread pieces: piece sums, an exclusive
// scan, and a walk of the one piece that crosses t.
template <typename T>
__device__ int locate(const Params &p, const Weights &w, long long lo, long long hi, u128 t,
                      const float2 *tab, u128 *s_u128, int *s_i) {
  const long long n = hi - lo;
  const long long per = (n + THREADS - 1) / THREADS;
  const long long t0 = lo + lmin(n, (long long)threadIdx.x * per), t1 = lmin(hi, t0 + per);
  u128 loc = 0;
  for (long long i = t0; i < t1; ++i) loc += weight<T>(p, w, i, tab);
  u128 tot;
  u128 cum = block_excl_u128<THREADS>(loc, tot, s_u128);
  int found = -1;
  if (cum <= t && t < cum + loc) {
    for (long long i = t0; i < t1; ++i) {
      cum += weight<T>(p, w, i, tab);
      if (cum > t) {
        found = (int)i;
        break;
      }
    }
  }
  return block_max_int<THREADS>(found, s_i);
}

template <typename T>
__global__ void __launch_bounds__(THREADS) icdf_kernel(const Params p) {
  __shared__ float2 tab[128];
  __shared__ u128 s_u128[THREADS / 32];
  __shared__ int s_i[THREADS / 32];
  __shared__ int s_last;
  __shared__ int s_c;
  pdl_wait();
  const int r = blockIdx.x / p.C2, c = blockIdx.x % p.C2;
  const Job jb = p.jobs[r];
  __shared__ uint64_t s_scale[2];
  Weights w;
  w.vp = row_view<T>(p, jb.prow);
  w.resid = jb.qrow >= 0;
  w.ap = w.aq = 0;
  if (w.resid) {
    w.vq = row_view<T>(p, jb.qrow);
    if (threadIdx.x == 0) {  // 2^124 / S: fp64 divisions, once per CTA
      s_scale[0] = __double2ull_rn(0x1p124 / u128_to_d(w.vp.S));
      s_scale[1] = __double2ull_rn(0x1p124 / u128_to_d(w.vq.S));
    }
  }
  load_table(tab);
  __syncthreads();
  if (w.resid) {
    w.ap = s_scale[0];
    w.aq = s_scale[1];
  }
  const long long lo = (long long)c * p.V / p.C2, hi = (long long)(c + 1) * p.V / p.C2;
  u128 loc = 0;
  for (long long i = lo + threadIdx.x; i < hi; i += THREADS) loc += weight<T>(p, w, i, tab);
  loc = block_sum_u128<THREADS>(loc, s_u128);
  uint64_t *part = p.ipart + ((size_t)r * p.C2 + c) * 2;
  if (threadIdx.x == 0) {
    part[0] = (uint64_t)loc;
    part[1] = (uint64_t)(loc >> 64);
  }
  if (!last_arriver(&p.icnt[r], (unsigned)p.C2, &s_last)) return;
  // the round's last CTA: chunk totals, the sample, then reset the round's rows
  __shared__ u128 s_part[acc::MAX_CHUNKS];
  const uint64_t *rp = p.ipart + (size_t)r * p.C2 * 2;
  for (int k = threadIdx.x; k < p.C2; k += THREADS)
    s_part[k] = ((u128)__ldcg(reinterpret_cast<const unsigned long long *>(rp + 2 * k + 1)) << 64) |
                __ldcg(reinterpret_cast<const unsigned long long *>(rp + 2 * k));
  __syncthreads();
  u128 W = 0;
  for (int k = 0; k < p.C2; ++k) W += s_part[k];
  int j;
  if (w.resid && W == 0) {
    // (p - q)+ vanishes: sample p itself
    w.resid = false;
    u128 Wp = 0;
    for (long long i = threadIdx.x; i < p.V; i += THREADS) Wp += weight<T>(p, w, i, tab);
    Wp = block_sum_u128<THREADS>(Wp, s_u128);
    u128 t = floor_mul(jb.u, Wp);
    if (t >= Wp) t = Wp - 1;
    j = locate<T>(p, w, 0, p.V, t, tab, s_u128, s_i);
  } else {
    u128 t = floor_mul(jb.u, W);
    if (t >= W) t = W - 1;
    // the chunk whose range of running sums holds t
    if (threadIdx.x == 0) {
      u128 cum = 0;
      int ck = p.C2 - 1;
      for (int k = 0; k < p.C2; ++k) {
        const u128 v = s_part[k];
        if (cum + v > t) {
          ck = k;
          break;
        }
        cum += v;
      }
      s_c = ck;
      s_u128[0] = cum;
    }
    __syncthreads();
    const int ck = s_c;
    const u128 base = s_u128[0];
    __syncthreads();
    j = locate<T>(p, w, (long long)ck * p.V / p.C2, (long long)(ck + 1) * p.V / p.C2, t - base, tab,
                  s_u128, s_i);
  }
  if (threadIdx.x == 0) p.out_tok[(size_t)r * (p.K + 1) + jb.pos] = j;
  // every pass of this call has read the round's rows: reset their sums
  const int rows2 = 2 * p.K + 1;
  for (int k = threadIdx.x; k < rows2; k += THREADS) {
    Hdr &h = hdr_of(p, (long long)r * rows2 + k);
    h.maxkey = 0u;
    h.z_lo = 0ull;
    h.z_hi = 0ull;
  }
}

// ----------------------------------------------------------------- host --
struct Layout {
  size_t hdr, jobs, icnt, ipart, hist, list, total;
};

Layout layout(int R, int K, int V, int C2) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = (size_t)R * (2 * K + 1);
  Layout L;
  L.hdr = 0;
  L.jobs = L.hdr + up(rows * HDR_BYTES);
  L.icnt = L.jobs + up((size_t)R * sizeof(Job));
  L.ipart = L.icnt + up((size_t)R * 4);
  L.hist = L.ipart + up((size_t)R * C2 * 16);
  const bool big = V > CAP;
  L.list = L.hist + (big ? up(rows * NB * 4) : 0);
  L.total = L.list + (big ? up(rows * CAP * 8) : 0);
  return L;
}

template <typename T>
sv_status launch_all(const Params &p, long long rows, cudaStream_t s) {
  const bool has_k = p.top_k > 0, has_p = p.top_p < 1.f;
  const dim3 gC((unsigned)(rows * p.C)), b(THREADS);
  const size_t hist_smem = (size_t)NB * 4;
  cudaError_t e = cudaSuccess;
  if (p.V <= CAP) {
    int P2 = 1;  // power of two >= V
    while (P2 < p.V) P2 <<= 1;
    e = launch(select_kernel<T, MODE_SMALL>, dim3((unsigned)rows), dim3(SEL_THREADS),
               (size_t)P2 * 16, s, p);
    if (e != cudaSuccess) return SV_ERR_CUDA;
  } else {
    e = launch(max_kernel<T>, gC, b, 0, s, p);
    if (e != cudaSuccess) return SV_ERR_CUDA;
    if (has_k) {
      e = launch(sum_kernel<T, COUNT_HIST>, gC, b, hist_smem, s, p);
      if (e == cudaSuccess) e = launch(compact_kernel<T, MODE_TOPK>, gC, b, 0, s, p);
      if (e == cudaSuccess)
        e = launch(select_kernel<T, MODE_TOPK>, dim3((unsigned)rows), dim3(SEL_THREADS),
                   (size_t)CAP * 8 + (size_t)SUB * 4, s, p);
      if (e != cudaSuccess) return SV_ERR_CUDA;
    }
    if (has_p) {
      e = launch(sum_kernel<T, SUM_HIST>, gC, b, hist_smem, s, p);
      if (e == cudaSuccess) e = launch(compact_kernel<T, MODE_TOPP>, gC, b, 0, s, p);
      if (e == cudaSuccess)
        e = launch(select_kernel<T, MODE_TOPP>, dim3((unsigned)rows), dim3(SEL_THREADS),
                   (size_t)CAP * 16 + (size_t)SUB * 4, s, p);
    } else {
      e = launch(sum_kernel<T, SUM_ONLY>, gC, b, 0, s, p);
    }
    if (e != cudaSuccess) return SV_ERR_CUDA;
  }
  e = launch(decide_kernel<T>, dim3((unsigned)p.R), dim3(32), 0, s, p);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  e = launch(icdf_kernel<T>, dim3((unsigned)(p.R * p.C2)), b, 0, s, p);
  return from_cuda(e);
}

}  // namespace whole

namespace acc {

static int icdf_chunks(int R, int V) { return chunks_per_row(R, V, device_sm_count()); }

size_t whole_workspace_bytes(int R, int K, int V) {
  if (R < 1 || K < 1 || V < 1) return 0;
  return whole::layout(R, K, V, icdf_chunks(R, V)).total;
}

sv_status whole_launch(const WholeArgs &a, cudaStream_t s) {
  using namespace whole;
  const long long rows = (long long)a.R * (2 * a.K + 1);
  if (rows > 0x7fffffffLL / MAX_CHUNKS || (long long)a.R * MAX_CHUNKS > 0x7fffffffLL)
    return SV_ERR_UNSUPPORTED;
  // log2(e) / T as float-float; very small temperatures would overflow it
  const double c = 1.4426950408889634 / (double)a.temperature;
  if (!(c <= 0x1p100)) return SV_ERR_UNSUPPORTED;
  const int sms = device_sm_count();
  const int C = chunks_per_row(rows, a.V, sms), C2 = icdf_chunks(a.R, a.V);
  const Layout L = layout(a.R, a.K, a.V, C2);
  if (!a.workspace || a.ws_bytes < L.total) return SV_ERR_WORKSPACE;
  uint8_t *w = static_cast<uint8_t *>(a.workspace);
  Params p{};
  p.tgt = a.tgt;
  p.drf = a.drf;
  p.drafts = a.drafts;
  p.u = a.u;
  p.out_tok = a.out_tok;
  p.out_n = a.out_n;
  p.R = a.R;
  p.K = a.K;
  p.V = a.V;
  p.C = C;
  p.C2 = C2;
  p.ch = (float)c;
  p.cl = (float)(c - (double)p.ch);
  p.top_k = a.top_k;
  p.top_p = a.top_p;
  p.hdr = w + L.hdr;
  p.jobs = reinterpret_cast<Job *>(w + L.jobs);
  p.icnt = reinterpret_cast<unsigned *>(w + L.icnt);
  p.ipart = reinterpret_cast<uint64_t *>(w + L.ipart);
  p.hist = reinterpret_cast<unsigned *>(w + L.hist);
  p.list = reinterpret_cast<uint64_t *>(w + L.list);
  return a.bf16 ? launch_all<__nv_bfloat16>(p, rows, s) : launch_all<float>(p, rows, s);
}

}  // namespace acc
}  // namespace sv
