/*
 * oracle.c -- plain, slow CPU oracle for the K-draft verify step of
 * multi-token-prediction speculative decoding.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or helper
 * with the CUDA library; the two meet only through seeded input tensors.
 *
 * Every floating-point step is carried in fp64 (the pages fix no precision).
 * Inputs arrive as the raw bytes the GPU path also receives: bf16 as uint16
 * bit patterns, packed 4-bit codes as uint32 words, logits as fp32.
 *
 * What each function computes, and where it is stated:
 *
 *  oracle_qmm   -- "The fastest way to run local LLMs on a Mac", section
 *                  "Decode is a memory-bandwidth problem" (one pass reads the
 *                  whole weight set) and "Speculative decoding and MTP on
 *                  Apple silicon", Facts (the small-M quantized matmul,
 *                  (M,5120)@(17408,5120)^T, 4-bit).  Weights are affine
 *                  group-quantised: w[n][k] = s[n][g]*q[n][k] + b[n][g],
 *                  g = k / group, q in 0..15 packed eight per uint32 word,
 *                  lowest k in the lowest nibble.  y[m][n] = sum_k x[m][k]*w[n][k].
 *
 *  oracle_gdn   -- GatedDeltaNet verify step with the previous round's commit
 *                  replayed from its tape (see the function).
 *
 *  oracle_qmm8  -- the 8-bit affine pack of the same pages ("Speculative
 *                  decoding and MTP on Apple silicon", Facts: skinny_qmm
 *                  flattens verify cost for 4-bit and 8-bit weights; 8-bit
 *                  is the sweet spot for the speedup ratio).  The same sum
 *                  with q in 0..255 packed four per uint32 word, lowest k in
 *                  the lowest byte.
 *
 *  oracle_attn  -- "Speculative decoding and MTP on Apple silicon", Facts
 *                  (attention verify with 2-8 query rows over the KV cache)
 *                  and "The fastest way ...", "Why token 1,000 is faster than
 *                  token 100,000" (each step reads the whole KV cache).
 *                  Row i of the M verify rows sits at cache slot L-M+i and
 *                  sees slots 0..L-M+i (causal among the drafts); query head
 *                  h reads KV head h / (Hq/Hkv).  Plain softmax attention.
 *
 *  oracle_attn_masked -- the same with a tree of drafts instead of a chain
 *                  ("Speculative decoding and MTP on Apple silicon", Facts:
 *                  ddtree-mlx verifies a draft tree with tree-attention
 *                  masks; ReDrafter's dynamic tree attention): row i sees
 *                  every slot before L-M and the draft slot L-M+j iff bit j
 *                  of mask[i] is set.  The chain is mask[i] = 2^(i+1) - 1.
 *
 *  oracle_dist / oracle_accept -- "The fastest way ...", section "Why exact
 *                  acceptance matters": accept a draft x with probability
 *                  min(1, p(x)/q(x)), on rejection resample from (p-q)+, which
 *                  reproduces the model's distribution at any temperature;
 *                  and "Speculative decoding and MTP on Apple silicon", Facts:
 *                  draft and verify distributions must be truncated the same
 *                  way (same top-k/top-p).  The steps follow those passages in
 *                  their order; readings where the pages are silent are listed
 *                  beside each step.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Planted-mistake switch for the pin tests: 0 = the oracle as specified.
 * A non-zero value makes one named step wrong on purpose so that a test can
 * show its pins catch that class of mistake.  Never set outside tests. */
static int g_mutant = 0;
void oracle_set_mutant(int m) { g_mutant = m; }

enum {
  MUT_NONE = 0,
  MUT_QMM_NIBBLE_HIGH_FIRST = 1, /* read the nibbles of a word high-first   */
  MUT_QMM_GROUP_OFF_BY_ONE = 2,  /* take scale/bias of group g+1 (clamped)  */
  MUT_QMM_DROP_BIAS = 3,         /* forget the bias term                    */
  MUT_ATTN_NO_CAUSAL = 4,        /* every row sees all L slots              */
  MUT_ATTN_MASK_OFF_BY_ONE = 5,  /* row i sees up to slot L-M+i-1           */
  MUT_ATTN_GQA_MODULO = 6,       /* kv head h % Hkv instead of h / group    */
  MUT_ACC_RESIDUAL_SIGN = 7,     /* resample from (q-p)+                    */
  MUT_ACC_REUSE_UNIFORM = 8,     /* final sample uses u_i instead of u_K    */
  MUT_ACC_NO_DRAFT_TRUNC = 9,    /* truncate the target only                */
  MUT_ACC_GREEDY = 10,           /* accept iff x == argmax p, emit argmax   */
  MUT_ACC_TOPP_INCLUSIVE = 11,   /* top-p keeps j iff mass above <= top_p   */
  MUT_ACC_NAIVE = 12,            /* sample y ~ p with u_i, accept iff y == x */
  MUT_ATTN_MASK_BIT_ORDER = 13,  /* draft slot j read from bit M-1-j        */
  MUT_QMM8_BYTE_HIGH_FIRST = 14, /* read the bytes of a word high-first     */
  MUT_QMM8_SIGNED = 15,          /* read 8-bit codes as signed (q - 256)    */
  MUT_DEPTH_NO_BONUS = 16,       /* tokens per round without the +1         */
  MUT_DEPTH_CONDITIONAL = 17,    /* multiply the acceptances again          */
  MUT_DEPTH_TIES_DEEPER = 18,    /* ties go to the larger depth             */
  MUT_GDN_NO_DECAY_IN_DELTA = 19,/* correction v - S k instead of v - a S k */
  MUT_GDN_OUTPUT_BEFORE = 20,    /* read o_t from the state before token t  */
  MUT_GDN_TRANSPOSED = 21,       /* S^T k instead of S k                    */
  MUT_GDN_HEAD_MODULO = 22,      /* key head h % Hk instead of h / (Hv/Hk)  */
};

static double bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static int omp_threads(int threads) {
#ifdef _OPENMP
  return threads > 0 ? threads : omp_get_max_threads();
#else
  (void)threads;
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Quantised small-M matmul                                                  */
/* ------------------------------------------------------------------------ */

/* Code q[n][k] of the canonical packing: word wq[n][k/8], nibble k%8 counted
 * from the least significant end. */
static unsigned code_at(const uint32_t *wq, int K, int n, int k) {
  uint32_t word = wq[(size_t)n * (size_t)(K / 8) + (size_t)(k / 8)];
  int nib = k % 8;
  if (g_mutant == MUT_QMM_NIBBLE_HIGH_FIRST) nib = 7 - nib;
  return (unsigned)((word >> (4 * nib)) & 15u);
}

/* 8-bit code q[n][k] of the canonical packing: word wq[n][k/4], byte k%4
 * counted from the least significant end, q in 0..255. */
static double code8_at(const uint32_t *wq, int K, int n, int k) {
  uint32_t word = wq[(size_t)n * (size_t)(K / 4) + (size_t)(k / 4)];
  int byte = k % 4;
  if (g_mutant == MUT_QMM8_BYTE_HIGH_FIRST) byte = 3 - byte;
  unsigned q = (word >> (8 * byte)) & 255u;
  if (g_mutant == MUT_QMM8_SIGNED && q >= 128u) return (double)q - 256.0;
  return (double)q;
}

/* y[m][n] (row-major [M][N]) = sum_k x[m][k] * (s[n][g]*q[n][k] + b[n][g]).
 * x: bf16 [M][K]; wq: uint32 [N][K/8]; scales, biases: bf16 [N][K/group].
 * Dequantised weights are exact in fp64; products and the running sum are
 * fp64.  Returns 0, or -1 on a shape the packing cannot hold. */
static int qmm_impl(const uint16_t *x, const uint32_t *wq, const uint16_t *scales,
                    const uint16_t *biases, int M, int N, int K, int group, int bits,
                    double *y, int threads) {
  if (M < 0 || N < 0 || K < 0 || group <= 0 || K % 8 != 0 || K % group != 0)
    return -1;
  const int G = K / group;
  double *xd = (double *)malloc(sizeof(double) * (size_t)M * (size_t)K + 1);
  if (!xd) return -1;
  for (size_t i = 0; i < (size_t)M * (size_t)K; ++i) xd[i] = bf16_to_double(x[i]);
  int failed = 0;
#pragma omp parallel num_threads(omp_threads(threads))
  {
    double *w = (double *)malloc(sizeof(double) * (size_t)K + 1);
    if (!w) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(static)
    for (int n = 0; n < N; ++n) {
      if (!w) continue;
      for (int k = 0; k < K; ++k) {
        int g = k / group;
        if (g_mutant == MUT_QMM_GROUP_OFF_BY_ONE && g + 1 < G) g = g + 1;
        double s = bf16_to_double(scales[(size_t)n * G + g]);
        double b = bf16_to_double(biases[(size_t)n * G + g]);
        if (g_mutant == MUT_QMM_DROP_BIAS) b = 0.0;
        const double q = bits == 8 ? code8_at(wq, K, n, k) : (double)code_at(wq, K, n, k);
        w[k] = s * q + b;
      }
      for (int m = 0; m < M; ++m) {
        const double *xm = xd + (size_t)m * K;
        double acc = 0.0;
        for (int k = 0; k < K; ++k) acc += xm[k] * w[k];
        y[(size_t)m * N + n] = acc;
      }
    }
    free(w);
  }
  free(xd);
  return failed ? -1 : 0;
}

int oracle_qmm(const uint16_t *x, const uint32_t *wq, const uint16_t *scales,
               const uint16_t *biases, int M, int N, int K, int group,
               double *y, int threads) {
  return qmm_impl(x, wq, scales, biases, M, N, K, group, 4, y, threads);
}

/* The 8-bit affine variant: the same sum with q[n][k] in 0..255 packed four
 * per uint32 word (wq: uint32 [N][K/4]), lowest k in the lowest byte. */
int oracle_qmm8(const uint16_t *x, const uint32_t *wq, const uint16_t *scales,
                const uint16_t *biases, int M, int N, int K, int group,
                double *y, int threads) {
  return qmm_impl(x, wq, scales, biases, M, N, K, group, 8, y, threads);
}

/* ------------------------------------------------------------------------ */
/* Multi-row verify attention                                                */
/* ------------------------------------------------------------------------ */

/* q: bf16 [M][Hq][D]; k, v: bf16 [Hkv][stride][D] (slot j of head g at row
 * g*stride + j); o: fp64 [M][Hq][D].  Row i (0..M-1) of the verify block is
 * the token in slot L-M+i and attends to slots 0..L-M+i.  Scores
 * s_j = scale * <q, k_j>, weights exp(s_j - max s) / sum, output
 * sum_j weight_j * v_j.  Returns 0, or -1 on bad arguments. */
/* Slot j visible to verify row i: the chain (mask NULL) or the draft mask. */
static int visible(const uint32_t *mask, int M, int i, int64_t L, int64_t j, int64_t last) {
  if (!mask) return j <= last;
  if (j < L - M) return 1;
  int bit = (int)(j - (L - M));
  if (g_mutant == MUT_ATTN_MASK_BIT_ORDER) bit = M - 1 - bit;
  return (int)((mask[i] >> bit) & 1u);
}

static int attn_impl(const uint16_t *q, const uint16_t *k, const uint16_t *v, int M,
                     int Hq, int Hkv, int D, int64_t L, int64_t stride, double scale,
                     const uint32_t *mask, double *o, int threads) {
  if (M <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0 || L < M ||
      stride < L || (mask && M > 32))
    return -1;
  const int group = Hq / Hkv;
  int failed = 0;
#pragma omp parallel num_threads(omp_threads(threads))
  {
    double *s = (double *)malloc(sizeof(double) * (size_t)L + 1);
    double *acc = (double *)malloc(sizeof(double) * (size_t)D + 1);
    if (!s || !acc) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int ih = 0; ih < M * Hq; ++ih) {
      if (!s || !acc) continue;
      const int i = ih / Hq, h = ih % Hq;
      int g = h / group;
      if (g_mutant == MUT_ATTN_GQA_MODULO) g = h % Hkv;
      int64_t last = L - M + i; /* newest visible slot of the chain */
      if (g_mutant == MUT_ATTN_NO_CAUSAL) last = L - 1;
      if (g_mutant == MUT_ATTN_MASK_OFF_BY_ONE) last = L - M + i - 1;
      const int64_t end = mask ? L - 1 : last; /* slots scanned: 0..end */
      const uint16_t *qr = q + ((size_t)i * Hq + h) * D;
      double smax = -INFINITY;
      for (int64_t j = 0; j <= end; ++j) {
        if (!visible(mask, M, i, L, j, last)) continue;
        const uint16_t *kr = k + ((size_t)g * stride + (size_t)j) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += bf16_to_double(qr[d]) * bf16_to_double(kr[d]);
        s[j] = scale * dot;
        if (s[j] > smax) smax = s[j];
      }
      double z = 0.0;
      for (int64_t j = 0; j <= end; ++j) {
        if (!visible(mask, M, i, L, j, last)) continue;
        s[j] = exp(s[j] - smax);
        z += s[j];
      }
      for (int d = 0; d < D; ++d) acc[d] = 0.0;
      for (int64_t j = 0; j <= end; ++j) {
        if (!visible(mask, M, i, L, j, last)) continue;
        const uint16_t *vr = v + ((size_t)g * stride + (size_t)j) * D;
        for (int d = 0; d < D; ++d) acc[d] += s[j] * bf16_to_double(vr[d]);
      }
      double *orow = o + ((size_t)i * Hq + h) * D;
      for (int d = 0; d < D; ++d) orow[d] = acc[d] / z;
    }
    free(s);
    free(acc);
  }
  return failed ? -1 : 0;
}

int oracle_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, int M,
                int Hq, int Hkv, int D, int64_t L, int64_t stride, double scale,
                double *o, int threads) {
  return attn_impl(q, k, v, M, Hq, Hkv, D, L, stride, scale, NULL, o, threads);
}

int oracle_attn_masked(const uint16_t *q, const uint16_t *k, const uint16_t *v, int M,
                       int Hq, int Hkv, int D, int64_t L, int64_t stride, double scale,
                       const uint32_t *mask, double *o, int threads) {
  if (!mask) return -1;
  return attn_impl(q, k, v, M, Hq, Hkv, D, L, stride, scale, mask, o, threads);
}

/* ------------------------------------------------------------------------ */
/* Exact acceptance                                                          */
/* ------------------------------------------------------------------------ */

typedef struct {
  double temperature;
  int top_k;
  double top_p;
} sampling_t;

/* Sort helpers: indices by (logit descending, index ascending). */
static _Thread_local const double *g_sort_key; /* per-thread sort key */
static int cmp_desc(const void *a, const void *b) {
  int ia = *(const int *)a, ib = *(const int *)b;
  double ka = g_sort_key[ia], kb = g_sort_key[ib];
  if (ka > kb) return -1;
  if (ka < kb) return 1;
  return (ia > ib) - (ia < ib);
}
static int cmp_double_desc(const void *a, const void *b) {
  double x = *(const double *)a, y = *(const double *)b;
  return (x < y) - (x > y);
}

/* The truncated sampling distribution of one logits row, written as a dense
 * fp64 vector p[0..V-1] (zero outside the support).
 *
 * Order of truncation (a reading: the pages say only "same top-p/top-k"):
 * temperature, then top-k, then top-p.
 *   T == 0: one-hot at the first index of the largest logit.
 *   l_j = z_j / T.
 *   0 < top_k < V: tau = k-th largest l counting repeats; keep l_j >= tau
 *     (every logit tied with the k-th is kept).
 *   softmax over the kept set: e_j = exp(l_j - max), Z summed in index order.
 *   top_p < 1: keep j iff the mass of kept tokens with a strictly larger
 *     logit is < top_p (ties kept together; the token that crosses top_p is
 *     kept).  Masses above are summed in decreasing-logit order; the new total
 *     is summed in index order and the kept p_j are divided by it.
 * Needs scratch of 2*V doubles + V ints.  Returns 0 or -1. */
static int dist_impl(const float *z, int V, sampling_t sp, double *p,
                     double *scratch, int *order) {
  if (V <= 0) return -1;
  if (sp.temperature == 0.0) {
    int best = 0;
    for (int j = 1; j < V; ++j)
      if (z[j] > z[best]) best = j;
    for (int j = 0; j < V; ++j) p[j] = 0.0;
    p[best] = 1.0;
    return 0;
  }
  double *l = scratch;       /* V */
  double *tmp = scratch + V; /* V */
  for (int j = 0; j < V; ++j) l[j] = (double)z[j] / sp.temperature;

  /* top-k threshold */
  double tau = -INFINITY;
  if (sp.top_k > 0 && sp.top_k < V) {
    memcpy(tmp, l, sizeof(double) * (size_t)V);
    qsort(tmp, (size_t)V, sizeof(double), cmp_double_desc);
    tau = tmp[sp.top_k - 1];
  }
  double lmax = -INFINITY;
  for (int j = 0; j < V; ++j)
    if (l[j] >= tau && l[j] > lmax) lmax = l[j];
  double Z = 0.0;
  for (int j = 0; j < V; ++j) {
    p[j] = (l[j] >= tau) ? exp(l[j] - lmax) : 0.0;
    Z += p[j];
  }
  for (int j = 0; j < V; ++j) p[j] = p[j] / Z;

  /* top-p (nucleus) */
  if (sp.top_p < 1.0) {
    int n = 0;
    for (int j = 0; j < V; ++j)
      if (l[j] >= tau) order[n++] = j;
    g_sort_key = l;
    qsort(order, (size_t)n, sizeof(int), cmp_desc);
    /* keep[j] stored in tmp as 1.0 / 0.0 */
    for (int j = 0; j < V; ++j) tmp[j] = 0.0;
    double above = 0.0; /* mass of strictly larger logits */
    int a = 0;
    while (a < n) {
      int b = a;
      while (b < n && l[order[b]] == l[order[a]]) ++b; /* tie group [a,b) */
      int keep = (g_mutant == MUT_ACC_TOPP_INCLUSIVE) ? (above <= sp.top_p)
                                                      : (above < sp.top_p);
      for (int c = a; c < b; ++c) tmp[order[c]] = keep ? 1.0 : 0.0;
      for (int c = a; c < b; ++c) above += p[order[c]];
      a = b;
    }
    double S = 0.0;
    for (int j = 0; j < V; ++j)
      if (tmp[j] != 0.0) S += p[j];
    for (int j = 0; j < V; ++j) p[j] = (tmp[j] != 0.0) ? p[j] / S : 0.0;
  }
  return 0;
}

int oracle_dist(const float *z, int V, double temperature, int top_k,
                double top_p, double *p) {
  if (V <= 0 || temperature < 0.0 || top_k < 0 || !(top_p > 0.0 && top_p <= 1.0))
    return -1;
  sampling_t sp = {temperature, top_k, top_p};
  double *scratch = (double *)malloc(sizeof(double) * 2 * (size_t)V);
  int *order = (int *)malloc(sizeof(int) * (size_t)V);
  int rc = (scratch && order) ? dist_impl(z, V, sp, p, scratch, order) : -1;
  free(scratch);
  free(order);
  return rc;
}

/* Inverse CDF in vocabulary order: the smallest j with sum_{i<=j} w_i > t;
 * if rounding leaves none, the largest j with w_j > 0. */
static int icdf(const double *w, int V, double t) {
  double c = 0.0;
  int last_pos = 0;
  for (int j = 0; j < V; ++j) {
    c += w[j];
    if (w[j] > 0.0) last_pos = j;
    if (c > t) return j;
  }
  return last_pos;
}

/* One speculative round per r in 0..R-1.
 *   zt: fp32 target logits [R][K+1][V] (rows 0..K-1 score the drafts, row K
 *       is the bonus row); zd: fp32 draft logits [R][K][V];
 *   drafts: int32 [R][K]; u: fp32 uniforms in [0,1) [R][K+1].
 *   out_tokens: int32 [R][K+1], -1 after the last emitted token;
 *   out_n: int32 [R], number of accepted drafts (0..K).
 * For i = 0..K-1, with p = dist(zt[i]), q = dist(zd[i]), x = drafts[i]:
 *   accept iff u_i * q(x) < p(x)   (probability min(1, p/q); a draft outside
 *     q's support is accepted iff p(x) > 0);
 *   else emit icdf(w, u_K * W) with w = max(p - q, 0), W = sum w (index
 *     order; W == 0 falls back to w = p, W = 1) and stop with n = i.
 * If all K are accepted, emit icdf(dist(zt[K]), u_K) and n = K.
 * u_K serves the one final sample (residual or bonus, never both). */
int oracle_accept(const float *zt, const float *zd, const int32_t *drafts,
                  const float *u, int R, int K, int V, double temperature,
                  int top_k, double top_p, int32_t *out_tokens, int32_t *out_n,
                  int threads) {
  if (R < 0 || K < 0 || V <= 0 || temperature < 0.0 || top_k < 0 ||
      !(top_p > 0.0 && top_p <= 1.0))
    return -1;
  sampling_t sp = {temperature, top_k, top_p};
  sampling_t sq = sp;
  if (g_mutant == MUT_ACC_NO_DRAFT_TRUNC) {
    sq.top_k = 0;
    sq.top_p = 1.0;
  }
  int failed = 0;
#pragma omp parallel num_threads(omp_threads(threads))
  {
    double *p = (double *)malloc(sizeof(double) * (size_t)V);
    double *q = (double *)malloc(sizeof(double) * (size_t)V);
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    double *scratch = (double *)malloc(sizeof(double) * 2 * (size_t)V);
    int *order = (int *)malloc(sizeof(int) * (size_t)V);
    if (!p || !q || !w || !scratch || !order) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int r = 0; r < R; ++r) {
      if (!p || !q || !w || !scratch || !order) continue;
      const float *zt_r = zt + (size_t)r * (size_t)(K + 1) * (size_t)V;
      const float *zd_r = zd + (size_t)r * (size_t)K * (size_t)V;
      const float *u_r = u + (size_t)r * (size_t)(K + 1);
      int32_t *tok = out_tokens + (size_t)r * (size_t)(K + 1);
      for (int i = 0; i <= K; ++i) tok[i] = -1;
      int n = K;
      int i;
      for (i = 0; i < K; ++i) {
        int x = drafts[(size_t)r * K + i];
        dist_impl(zt_r + (size_t)i * V, V, sp, p, scratch, order);
        dist_impl(zd_r + (size_t)i * V, V, sq, q, scratch, order);
        double px = (x >= 0 && x < V) ? p[x] : 0.0;
        double qx = (x >= 0 && x < V) ? q[x] : 0.0;
        int accept;
        if (g_mutant == MUT_ACC_GREEDY) {
          int am = 0;
          for (int j = 1; j < V; ++j)
            if (p[j] > p[am]) am = j;
          accept = (x == am);
          if (!accept) {
            tok[i] = am;
            n = i;
            break;
          }
        } else if (g_mutant == MUT_ACC_NAIVE) {
          int y = icdf(p, V, (double)u_r[i]);
          accept = (y == x);
          if (!accept) {
            tok[i] = y;
            n = i;
            break;
          }
        } else {
          accept = ((double)u_r[i] * qx < px);
        }
        if (accept) {
          tok[i] = x;
          continue;
        }
        double W = 0.0;
        for (int j = 0; j < V; ++j) {
          double d = (g_mutant == MUT_ACC_RESIDUAL_SIGN) ? q[j] - p[j] : p[j] - q[j];
          w[j] = d > 0.0 ? d : 0.0;
          W += w[j];
        }
        if (W == 0.0) {
          memcpy(w, p, sizeof(double) * (size_t)V);
          W = 1.0;
        }
        double uf = (g_mutant == MUT_ACC_REUSE_UNIFORM) ? (double)u_r[i] : (double)u_r[K];
        tok[i] = icdf(w, V, uf * W);
        n = i;
        break;
      }
      if (i == K) {
        dist_impl(zt_r + (size_t)K * V, V, sp, p, scratch, order);
        if (g_mutant == MUT_ACC_GREEDY) {
          int am = 0;
          for (int j = 1; j < V; ++j)
            if (p[j] > p[am]) am = j;
          tok[K] = am;
        } else {
          tok[K] = icdf(p, V, (double)u_r[K]);
        }
        n = K;
      }
      out_n[r] = n;
    }
    free(p);
    free(q);
    free(w);
    free(scratch);
    free(order);
  }
  return failed ? -1 : 0;
}

/* ------------------------------------------------------------------------ */
/* Draft depth from measured cost curves                                     */
/* ------------------------------------------------------------------------ */

/* "Speculative decoding and MTP on Apple silicon", Facts: mlx-dspark
 * measures the verify and drafter cost curves once and picks the draft cap
 * from them; MTPLX keeps a depth only if it beats plain decoding.
 *
 * verify_us[K] (K = 0..Kmax): cost of a verify pass with K+1 rows (K = 0 is
 * the plain decode step); draft_us[K]: cost of drafting K tokens (NULL: 0);
 * accept[i-1] (i = 1..Kmax): probability that at least the first i drafts
 * of a round are accepted.  A round at depth K yields one token more than
 * the drafts it accepts, so its expected yield is 1 + sum_{i<=K} accept[i-1]
 * tokens at a cost of verify_us[K] + draft_us[K].  The result is the depth
 * whose yield per microsecond is highest, taken only when it is strictly
 * higher than plain decoding's 1 / verify_us[0]; among equal rates the
 * shallower depth wins.  rates[K] receives each depth's tokens per
 * microsecond.  Returns -1 on invalid input. */
int oracle_pick_depth(const double *verify_us, const double *draft_us, const double *accept,
                      int Kmax, double *rates) {
  if (Kmax < 0 || !verify_us || (Kmax > 0 && !accept)) return -1;
  for (int K = 0; K <= Kmax; ++K) {
    const double d = draft_us ? draft_us[K] : 0.0;
    if (!(verify_us[K] > 0.0) || !(verify_us[K] < INFINITY)) return -1;
    if (!(d >= 0.0) || !(d < INFINITY)) return -1;
  }
  for (int i = 1; i <= Kmax; ++i) {
    if (!(accept[i - 1] >= 0.0 && accept[i - 1] <= 1.0)) return -1;
    if (i > 1 && accept[i - 1] > accept[i - 2]) return -1;
  }
  int best = 0;
  double best_rate = 0.0;
  for (int K = 0; K <= Kmax; ++K) {
    double tokens = (g_mutant == MUT_DEPTH_NO_BONUS) ? 0.0 : 1.0;
    double prod = 1.0;
    for (int i = 1; i <= K; ++i) {
      prod *= accept[i - 1];
      tokens += (g_mutant == MUT_DEPTH_CONDITIONAL) ? prod : accept[i - 1];
    }
    if (K == 0 && g_mutant == MUT_DEPTH_NO_BONUS) tokens = 1.0;
    const double cost = verify_us[K] + (draft_us ? draft_us[K] : 0.0);
    const double rate = tokens / cost;
    if (rates) rates[K] = rate;
    const int better = (g_mutant == MUT_DEPTH_TIES_DEEPER) ? rate >= best_rate : rate > best_rate;
    if (K == 0 || better) {
      best = K;
      best_rate = rate;
    }
  }
  return best;
}

/* ------------------------------------------------------------------------ */
/* GatedDeltaNet verify step with deferred commit (tape replay)              */
/* ------------------------------------------------------------------------ */

/* "Speculative decoding and MTP on Apple silicon", Facts: most layers of the
 * hybrid targets are GatedDeltaNet layers whose recurrent state is a fixed
 * size array that cannot be trimmed after a rejected draft; MTPLX rolls it
 * back with an "innovation tape" replayed in its GDN kernel.  The pages give
 * no recurrence; this is the published gated delta rule, per value head h
 * with state S (dv x dk) and key head g = h / (Hv/Hk):
 *     S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,  a_t = exp(g_t),
 *     o_t = S_t q_t.
 * One call first commits the previous round: the first n_replay tokens of
 * its tape (its k, v, g, b) are applied to `state` in place; then the M rows
 * of this round run from that state, giving o[M][Hv][dv], without touching
 * `state` (the next call commits them once acceptance is known).
 * state: fp64 [Hv][dv][dk]; tape_k: bf16 [n][Hk][dk]; tape_v: bf16 [n][Hv][dv];
 * tape_g, tape_b: fp32 [n][Hv]; q, k: bf16 [M][Hk][dk]; v: bf16 [M][Hv][dv];
 * g, b: fp32 [M][Hv]. */
static void gdn_token(double *S, int dv, int dk, const double *kk, const double *vv, double a,
                      double b) {
  for (int i = 0; i < dv; ++i) {
    double u = 0.0;
    for (int j = 0; j < dk; ++j)
      u += (g_mutant == MUT_GDN_TRANSPOSED ? S[(size_t)j * dk + i] : S[(size_t)i * dk + j]) * kk[j];
    const double delta = (g_mutant == MUT_GDN_NO_DECAY_IN_DELTA) ? vv[i] - u : vv[i] - a * u;
    for (int j = 0; j < dk; ++j) S[(size_t)i * dk + j] = a * S[(size_t)i * dk + j] + b * delta * kk[j];
  }
}

int oracle_gdn(double *state, const uint16_t *tape_k, const uint16_t *tape_v, const float *tape_g,
               const float *tape_b, int n_replay, const uint16_t *q, const uint16_t *k,
               const uint16_t *v, const float *g, const float *b, int M, int Hk, int Hv, int dk,
               int dv, double *o, int threads) {
  if (M < 0 || n_replay < 0 || Hk < 1 || Hv < 1 || Hv % Hk != 0 || dk < 1 || dv < 1) return -1;
  if (g_mutant == MUT_GDN_TRANSPOSED && dk != dv) return -1;
  const int grp = Hv / Hk;
  int failed = 0;
#pragma omp parallel num_threads(omp_threads(threads))
  {
    double *kk = (double *)malloc(sizeof(double) * (size_t)dk);
    double *qq = (double *)malloc(sizeof(double) * (size_t)dk);
    double *vv = (double *)malloc(sizeof(double) * (size_t)dv);
    double *S = (double *)malloc(sizeof(double) * (size_t)dv * dk);
    if (!kk || !qq || !vv || !S) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(static)
    for (int h = 0; h < Hv; ++h) {
      if (!kk || !qq || !vv || !S) continue;
      const int hk = (g_mutant == MUT_GDN_HEAD_MODULO) ? h % Hk : h / grp;
      double *Sh = state + (size_t)h * dv * dk;
      for (int t = 0; t < n_replay; ++t) {  /* commit the previous round */
        for (int j = 0; j < dk; ++j) kk[j] = bf16_to_double(tape_k[((size_t)t * Hk + hk) * dk + j]);
        for (int i = 0; i < dv; ++i) vv[i] = bf16_to_double(tape_v[((size_t)t * Hv + h) * dv + i]);
        gdn_token(Sh, dv, dk, kk, vv, exp((double)tape_g[(size_t)t * Hv + h]),
                  (double)tape_b[(size_t)t * Hv + h]);
      }
      memcpy(S, Sh, sizeof(double) * (size_t)dv * dk);
      for (int t = 0; t < M; ++t) {  /* this round's rows, from a copy */
        for (int j = 0; j < dk; ++j) {
          kk[j] = bf16_to_double(k[((size_t)t * Hk + hk) * dk + j]);
          qq[j] = bf16_to_double(q[((size_t)t * Hk + hk) * dk + j]);
        }
        for (int i = 0; i < dv; ++i) vv[i] = bf16_to_double(v[((size_t)t * Hv + h) * dv + i]);
        double *ot = o + ((size_t)t * Hv + h) * dv;
        if (g_mutant == MUT_GDN_OUTPUT_BEFORE)
          for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * qq[j];
            ot[i] = acc;
          }
        gdn_token(S, dv, dk, kk, vv, exp((double)g[(size_t)t * Hv + h]), (double)b[(size_t)t * Hv + h]);
        if (g_mutant != MUT_GDN_OUTPUT_BEFORE)
          for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * qq[j];
            ot[i] = acc;
          }
      }
    }
    free(kk);
    free(qq);
    free(vv);
    free(S);
  }
  return failed ? -1 : 0;
}
