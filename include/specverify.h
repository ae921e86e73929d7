/*
 * specverify.h -- C ABI of libspecverify.so, the K-draft verify step of
 * multi-token-prediction (MTP) speculative decoding on one GB300 (sm_103a).
 *
 * One verify pass scores the last committed token plus K drafted tokens as
 * M = K+1 rows in a single forward pass, so every weight byte and every KV
 * byte is read once for all rows ("The fastest way to run local LLMs on a
 * Mac", sections "Decode is a memory-bandwidth problem" and "Why native MTP
 * doubles decode").  The library provides the three data-parallel pieces of
 * that pass:
 *
 *   qmm_small_m  -- small-M matmul over 4-bit group-quantised weights
 *                   (qmm8_small_m: the same over 8-bit weights)
 *   verify_attn  -- multi-row decode attention over a bf16 GQA KV cache
 *   spec_accept  -- exact Leviathan-Chen acceptance of the drafts
 *
 * Conventions shared by every entry point
 *   - Pointers marked "device" are caller-owned device memory on the current
 *     CUDA device; the library never allocates, frees or keeps them.
 *   - Every compute call is asynchronous on `stream` (NULL = legacy default
 *     stream) and launches only the library's own kernels.
 *   - Arguments are checked on the host before anything is launched; a
 *     rejected call launches nothing and returns a non-zero sv_status.  There
 *     is no fallback path of any kind.
 *   - Scratch memory is passed in by the caller (`workspace`, `ws_bytes`);
 *     size it with the matching *_workspace_bytes query.  Workspaces must be
 *     zero-filled once before their first use (every call leaves them ready
 *     for the next); one workspace must not be shared by calls that may run
 *     concurrently.
 *   - Device-side bounded waits that expire set a device error word that
 *     sv_last_device_error() reports as SV_ERR_TIMEOUT; no kernel ever spins
 *     without a limit.
 *   - Results are deterministic for fixed inputs (no floating-point atomics;
 *     split plans depend only on shapes and the device's SM count).
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported symbols of the shared library. */
#if defined(__GNUC__)
#define SV_API __attribute__((visibility("default")))
#else
#define SV_API
#endif

/* Same type as cudaStream_t; declared here so that callers need no CUDA
 * header. */
typedef struct CUstream_st *sv_stream_t;

typedef enum {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1, /* null pointer, negative size, inconsistent shape */
  SV_ERR_UNSUPPORTED = 2, /* well-formed but outside the supported shapes     */
  SV_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed           */
  SV_ERR_TIMEOUT = 4,     /* a bounded device-side wait expired               */
  SV_ERR_WORKSPACE = 5,   /* workspace missing or smaller than required       */
  SV_ERR_OVERFLOW = 6     /* a candidate set outgrew its buffer (top-k ties)  */
} sv_status;

typedef enum { SV_BF16 = 0, SV_F32 = 1 } sv_dtype;

/* Sampling settings applied identically to the target and the draft rows
 * ("Speculative decoding and MTP on Apple silicon", Facts: the draft and
 * verify distributions must be truncated the same way).
 *   temperature >= 0 (0 = greedy one-hot at the first maximal logit);
 *   top_k >= 0 (0 = off; ties with the k-th largest logit are all kept);
 *   0 < top_p <= 1 (1 = off; a token is kept while the mass of strictly more
 *   likely kept tokens is below top_p). */
typedef struct {
  float temperature;
  int32_t top_k;
  float top_p;
} sv_sampling_params;

/* ---------------------------------------------------------------------- */
/* Quantised small-M matmul                                                 */
/* ---------------------------------------------------------------------- */
/*
 * y[m][n] = sum_k x[m][k] * (s[n][g] * q[n][k] + b[n][g]),  g = k / group.
 * The small-M quantized matmul of "Speculative decoding and MTP on Apple
 * silicon", Facts ((M,5120)@(17408,5120)^T at 4 bits, M = 2..16 verify rows):
 * each weight byte is streamed from HBM once for all M rows and dequantised
 * in registers; accumulation is fp32.
 *
 * Canonical weight layout (input to qmm_prepack):
 *   wq      uint32 [N][K/8]  eight 4-bit codes per word, code k%8 in bits
 *                            4*(k%8) .. 4*(k%8)+3 (lowest k lowest);
 *   scales  bf16   [N][K/group];
 *   biases  bf16   [N][K/group].
 * Supported: group == 64, K % 64 == 0, 1 <= M <= 16, N >= 1, K >= 64.
 */

/* Bytes of the prepacked weight buffer for an N x K matrix (0 if the shape
 * is unsupported).  Equal to N'*K/2 + N'*K/group*4 with N' = N rounded up
 * to 128: codes plus scales (stored times the kernel's power-of-two factors,
 * exactly) and biases, interleaved in batches of eight 16-row tiles (rows
 * N..N'-1 are zero). */
SV_API size_t qmm_packed_bytes(int N, int K, int group);

/* One-time relayout of canonical weights (device) into the opaque tiled
 * layout that qmm_small_m streams.  packed_out (device, at least
 * qmm_packed_bytes bytes, 16-byte aligned) receives the result; rows N..N'-1
 * are zero.  Asynchronous on `stream`. */
SV_API sv_status qmm_prepack(const uint32_t *wq, const void *scales, const void *biases,
                      int N, int K, int group, void *packed_out,
                      size_t packed_bytes, sv_stream_t stream);

/* Workspace bytes for qmm_small_m (partial sums of tile batches shared by
 * several CTAs, and per-batch arrival counters).  Depends on N, K and the
 * device's SM count. */
SV_API size_t qmm_workspace_bytes(int M, int N, int K);

/* x: device bf16 [M][K] row-major, 16-byte aligned.
 * packed_w: device, from qmm_prepack for the same N, K, group (16-byte
 *   aligned).
 * y: device [M][N] row-major, bf16 (y_dtype SV_BF16) or fp32 (SV_F32).
 * workspace: device, >= qmm_workspace_bytes(M, N, K) bytes, zeroed once. */
SV_API sv_status qmm_small_m(const void *x_bf16, const void *packed_w, void *y,
                      sv_dtype y_dtype, int M, int N, int K, int group,
                      void *workspace, size_t ws_bytes, sv_stream_t stream);

/* The 8-bit affine variant ("Speculative decoding and MTP on Apple silicon",
 * Facts: skinny_qmm flattens the verify cost of 4-bit and 8-bit weights; 8-bit
 * is the sweet spot for the speedup ratio):
 *   y[m][n] = sum_k x[m][k] * (s[n][g] * q[n][k] + b[n][g]),  q in 0..255.
 * Canonical weight layout (input to qmm8_prepack):
 *   wq      uint32 [N][K/4]  four 8-bit codes per word, code k%4 in bits
 *                            8*(k%4) .. 8*(k%4)+7 (lowest k lowest);
 *   scales, biases as for qmm_small_m.
 * Supported shapes, argument rules, ownership and errors are those of the
 * 4-bit calls above.  The prepacked buffer (qmm8_packed_bytes = N'*K +
 * N'*K/group*4 bytes, N' = N rounded up to 128) is not interchangeable with
 * the 4-bit one.  Each code enters the tensor cores whole, as the fp16 value
 * 1024 + q (exact), against the same activations; a byte of weights holds one
 * code instead of two, so it costs the consumers less than at 4 bits. */
SV_API size_t qmm8_packed_bytes(int N, int K, int group);
SV_API sv_status qmm8_prepack(const uint32_t *wq, const void *scales, const void *biases,
                       int N, int K, int group, void *packed_out,
                       size_t packed_bytes, sv_stream_t stream);
SV_API size_t qmm8_workspace_bytes(int M, int N, int K);
SV_API sv_status qmm8_small_m(const void *x_bf16, const void *packed_w, void *y,
                       sv_dtype y_dtype, int M, int N, int K, int group,
                       void *workspace, size_t ws_bytes, sv_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Multi-row verify attention                                               */
/* ---------------------------------------------------------------------- */
/*
 * For verify row i in 0..M-1 and query head h in 0..Hq-1:
 *   O[i][h] = softmax_j( scale * <Q[i][h], K[g][j]> ) . V[g][j],
 *   j = 0 .. kv_len-M+i,  g = h / (Hq/Hkv).
 * The M verify rows are the newest M cache slots (the cache already holds
 * them), so draft row i sees the committed prefix and drafts 0..i: causal
 * among the drafts.  Each KV tile is read from HBM once for all M rows and
 * all Hq/Hkv query heads of its group ("Speculative decoding and MTP on
 * Apple silicon", Facts: a multi-row attention kernel reads each KV tile
 * once; flash-decoding verify kernel).  Softmax and accumulation are fp32.
 *
 * q: device bf16 [M][Hq][D]; o: device bf16 [M][Hq][D].
 * k_cache, v_cache: device bf16 [Hkv][kv_stride_tokens][D] (head-major; slot
 *   j of head g at element (g*kv_stride_tokens + j)*D), 16-byte aligned.
 * Supported: D in {128, 256}; Hq % Hkv == 0; 1 <= M; M*(Hq/Hkv) <= 96
 *   (e.g. M = 16 drafts at 6 query heads per KV head);
 *   M <= kv_len <= kv_stride_tokens; scale > 0 and finite.
 */
SV_API size_t verify_attn_workspace_bytes(int M, int Hq, int Hkv, int D, int64_t kv_len);

SV_API sv_status verify_attn(const void *q, const void *k_cache, const void *v_cache,
                      void *o, int M, int Hq, int Hkv, int D, int64_t kv_len,
                      int64_t kv_stride_tokens, float scale, void *workspace,
                      size_t ws_bytes, sv_stream_t stream);

/* verify_attn over a tree of drafts instead of a chain ("Speculative
 * decoding and MTP on Apple silicon", Facts: ddtree-mlx verifies a draft
 * tree with tree-attention masks; ReDrafter's dynamic tree attention).
 * Row i sees every slot before kv_len-M, and draft slot kv_len-M+j iff bit j
 * of draft_mask[i] is set (a node sees its ancestors and itself; the chain
 * of verify_attn is draft_mask[i] = 2^(i+1) - 1).
 * draft_mask: device uint32 [M], 4-byte aligned, read after the stream's
 *   previous work.  Supported: M <= 32, and everything verify_attn
 *   supports; the workspace is verify_attn_workspace_bytes().  A row that
 *   sees no slot at all (kv_len == M and draft_mask[i] == 0) has no defined
 *   output. */
SV_API sv_status verify_attn_masked(const void *q, const void *k_cache, const void *v_cache,
                             void *o, int M, int Hq, int Hkv, int D, int64_t kv_len,
                             int64_t kv_stride_tokens, float scale,
                             const uint32_t *draft_mask, void *workspace,
                             size_t ws_bytes, sv_stream_t stream);

/* verify_attn for callers that cannot allocate device memory -- a plugin
 * running inside another engine's enqueue call, code between the begin and
 * end of a stream capture where cudaMalloc is not allowed, or a service whose
 * device-memory budget is fixed at start-up.  (The pages have no counterpart;
 * this is an integration variant of verify_attn.)
 *
 * Same arguments, layouts, checks, kernels and results as verify_attn (the
 * two share one implementation), minus the workspace: the split-KV partials
 * live in one fixed 16 MiB array inside the library, which every GPU that
 * loads the library holds until the process exits.  The call allocates
 * nothing (no cudaMalloc/cudaFree or allocating library routine).  A shape
 * whose partials would exceed 16 MiB (verify_attn_workspace_bytes > 16 MiB)
 * is rejected with SV_ERR_WORKSPACE before anything is launched.  The
 * partials take 16 rows x (D + 2) floats per head segment for every 16 query
 * rows of a KV head, about two segments per SM: on 152 SMs with 24 query and
 * 4 KV heads at D = 256, M <= 8 fits (15.1 MB at M = 8) and M >= 9 is
 * refused; at D = 128 every supported M fits.
 *
 * The first call on each device looks up the array's device address (with
 * that device current); make that first call before any stream capture.
 * Every call shares the one array and nothing in it needs to start at zero
 * (each call writes all the partials it reads); calls whose kernels may
 * overlap on the GPU -- on different streams, or on different threads without
 * ordering -- race on it and must be serialised by the caller.  The device
 * address is kept for the life of the process: do not call this entry point
 * across a cudaDeviceReset() of that device (the same holds for the device
 * error word of every entry point). */
SV_API sv_status verify_attn_noalloc(const void *q, const void *k_cache,
                                     const void *v_cache, void *o, int M, int Hq,
                                     int Hkv, int D, int64_t kv_len,
                                     int64_t kv_stride_tokens, float scale,
                                     sv_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Exact acceptance                                                         */
/* ---------------------------------------------------------------------- */
/*
 * R independent speculative rounds of K drafts each ("The fastest way to run
 * local LLMs on a Mac", section "Why exact acceptance matters"; "Speculative
 * decoding and MTP on Apple silicon", Facts: Leviathan-Chen rejection
 * sampling with identical truncation).  For round r, with p_i the truncated
 * target distribution of row i and q_i that of draft row i:
 *   for i = 0..K-1: accept x = draft_tokens[r][i] iff u_i * q_i(x) < p_i(x);
 *   on the first rejection emit icdf((p_i - q_i)+, u_K) and stop;
 *   if all K are accepted emit icdf(p_K, u_K) (the bonus token).
 * icdf(w, u) is the first vocabulary index whose running sum of w exceeds
 * u * sum(w).  Truncation order: temperature, top-k, top-p.
 *
 * Two evaluation paths give the same decisions as the CPU definition (fp64
 * in the pages' order) except when a decision's margin is within rounding
 * (relative ~1e-13):
 *   - temperature 0, or 0 < top_k <= 1024 with top_k < V: the top-k set is
 *     selected exactly, and its distribution, the ratio test and the inverse
 *     CDF are evaluated in fp64 in the CPU definition's order;
 *   - every other setting with temperature > 0 (top_k = 0 or >= V: no top-k;
 *     top_k > 1024): the whole vocabulary.  exp(z/T - zmax/T) is computed in
 *     float-float arithmetic (relative error ~3e-14) and rounded to an
 *     integer with 62 fractional bits; the normaliser, the masses walked by
 *     top-p and the inverse CDF's running sums are exact integer sums of
 *     those values.  Tokens whose weight is below 2^-63 of the largest count
 *     as zero.
 * Results are deterministic on both paths.
 *
 * target_logits: device [R][K+1][V]; draft_logits: device [R][K][V]; dtype
 *   SV_F32 or SV_BF16 (both the same type); logits must not be NaN or +inf
 *   (-inf is a token of weight zero), and every row needs a finite logit.
 * draft_tokens: device int32 [R][K]; uniforms: device fp32 [R][K+1] in [0,1).
 * out_tokens: device int32 [R][K+1], -1 after the last emitted token.
 * out_num_accepted: device int32 [R], 0..K.
 * Supported: 1 <= K <= 32, V >= 1, any top_k >= 0; temperature 0 or
 *   log2(e)/temperature <= 2^100 (temperature >= about 1.2e-30).  On the
 *   candidate-list path a top-k set enlarged by ties beyond 2048 entries is
 *   reported as SV_ERR_OVERFLOW by sv_last_device_error() and its round's
 *   out_num_accepted is -1; the whole-vocabulary path has no such limit.
 * workspace: device, >= spec_accept_workspace_bytes(R, K, V) bytes, zeroed
 *   once (it covers both paths; about 110 KB per logits row for V > 4096).
 *   After a call that returned an error, zero it again.
 */
SV_API size_t spec_accept_workspace_bytes(int R, int K, int V);

SV_API sv_status spec_accept(const void *target_logits, const void *draft_logits,
                      sv_dtype logit_dtype, const int32_t *draft_tokens,
                      const float *uniforms, sv_sampling_params params, int R,
                      int K, int V, int32_t *out_tokens,
                      int32_t *out_num_accepted, void *workspace,
                      size_t ws_bytes, sv_stream_t stream);

/* ---------------------------------------------------------------------- */
/* lm_head fused with the acceptance's vocabulary scan                      */
/* ---------------------------------------------------------------------- */
/* The verify pass ends with the lm_head (hidden -> vocabulary logits) and the
 * acceptance, whose first step reads every logit again to select the top-k
 * ("The fastest way to run local LLMs on a Mac", sections "Why native MTP
 * doubles decode" and "Why exact acceptance matters").  Three calls split
 * that work so that only what depends on the target logits follows the
 * lm_head:
 *   qmm_small_m_topk: qmm_small_m with fp32 output plus the selection in its
 *     epilogue: each CTA, holding whole 128-column batches of the vocabulary,
 *     writes per logits row the top-k of its own columns (every logit equal
 *     to the k-th largest kept) while its logits are on chip;
 *   spec_accept_draft_select: the draft rows' top-k and truncated
 *     distributions from draft logits into the acceptance workspace (the
 *     draft logits exist before the verify pass);
 *   spec_accept_lists: the target rows' sets merged from the lists -- and
 *     the draft rows' too when the drafter's own lm_head (the MTP head ends
 *     in the same vocabulary projection) made lists with qmm_small_m_topk --
 *     their distributions, and the accept / residual / bonus chain.
 * The outputs equal spec_accept on the same logits, bit for bit.
 *
 * Supported: the candidate-list settings of spec_accept (temperature 0, or
 * 0 < top_k <= 1024 with top_k < N); N of at least 128 columns per SM (the
 * launch keeps whole batches per CTA: a 152064-token vocabulary qualifies, a
 * 5120-column projection does not), 1 <= M <= 16; everything else is
 * SV_ERR_UNSUPPORTED.
 *
 * qmm_small_m_topk: arguments of qmm_small_m with y fp32 [M][N] (device,
 *   written as by qmm_small_m), params the sampling settings of the
 *   acceptance that will read the lists, lists (device, 16-byte aligned, at
 *   least qmm_topk_lists_bytes(M, N, K) bytes; opaque: a header, then per
 *   (row, CTA) a count, keys and indices), and the workspace of qmm_small_m.
 * spec_accept_draft_select: draft_logits [R][K][V] (device, SV_F32 or
 *   SV_BF16), the sampling settings, and the workspace of spec_accept (R, K,
 *   V), which spec_accept_lists then reads: order the two calls on one
 *   stream or with an event.
 * spec_accept_lists: target_lists from qmm_small_m_topk over M = R*(K+1)
 *   rows (round r's row j is lm_head row r*(K+1) + j) made with the same
 *   params; draft_lists likewise over the drafter's M = R*K rows (round r's
 *   draft i is row r*K + i), or NULL when spec_accept_draft_select has
 *   filled the workspace (order the two calls on one stream or with an
 *   event); draft_tokens, uniforms, outputs as in spec_accept.  Lists made
 *   for fewer rows or a smaller top-k are reported by sv_last_device_error()
 *   as SV_ERR_INVALID_ARG, with out_num_accepted -1 for the rounds concerned. */
SV_API size_t qmm_topk_lists_bytes(int M, int N, int K);
SV_API sv_status qmm_small_m_topk(const void *x_bf16, const void *packed_w, float *y, int M, int N,
                                  int K, int group, sv_sampling_params params, void *lists,
                                  size_t lists_bytes, void *workspace, size_t ws_bytes,
                                  sv_stream_t stream);
SV_API sv_status spec_accept_draft_select(const void *draft_logits, sv_dtype logit_dtype,
                                          sv_sampling_params params, int R, int K, int V,
                                          void *workspace, size_t ws_bytes, sv_stream_t stream);
SV_API sv_status spec_accept_lists(const void *target_lists, const void *draft_lists,
                                   const int32_t *draft_tokens, const float *uniforms,
                                   sv_sampling_params params, int R, int K, int V,
                                   int32_t *out_tokens, int32_t *out_num_accepted, void *workspace,
                                   size_t ws_bytes, sv_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Status and launch control                                                */
/* ---------------------------------------------------------------------- */

/* Static description of a status code (never NULL). */
SV_API const char *sv_status_string(sv_status status);

/* ---------------------------------------------------------------------- */
/* GatedDeltaNet verify step with deferred commit                           */
/* ---------------------------------------------------------------------- */
/* The recurrent layers of a hybrid target ("Speculative decoding and MTP on
 * Apple silicon", Facts: GDN state is a fixed-size array that cannot be
 * trimmed after a rejected draft; MTPLX replays an "innovation tape" in its
 * GDN kernel).  Per value head h with key head g = h / (Hv/Hk) and state S
 * (dv x dk), each token applies the gated delta rule
 *     S <- exp(gt) S (I - bt k k^T) + bt v k^T   and reads   o = S q.
 * One call (1) commits the previous round: its first n_replay tokens (the
 * tape: that round's own k, v, g, beta) are applied to `state` in place, and
 * (2) runs this round's M rows from the committed state without writing it,
 * giving o.  After acceptance of n drafts, the next call passes this round's
 * k, v, g, beta as its tape with n_replay = n + 1 (the round's first row and
 * its n accepted drafts).  M = 0 only commits.
 * state: device fp32 [Hv][dv][dk], 16-byte aligned, read and (if n_replay >
 *   0) written.
 * tape_k: device bf16 [>= n_replay][Hk][dk]; tape_v: bf16 [>= n_replay][Hv][dv];
 *   tape_g, tape_beta: fp32 [>= n_replay][Hv]; NULL allowed when n_replay = 0.
 * q, k: device bf16 [M][Hk][dk] (normalised by the caller); v: bf16 [M][Hv][dv];
 *   g (log decay), beta: fp32 [M][Hv]; o: [M][Hv][dv], bf16 or fp32 (o_dtype).
 * q, k, tape_k 16-byte aligned.  Supported: dk in {64, 128, 256}; Hv % Hk == 0;
 *   n_replay <= 64 and M <= 64 (SV_ERR_UNSUPPORTED beyond).
 * fp32 arithmetic throughout.  Asynchronous on `stream`; calls on one state
 * must be ordered. */
SV_API sv_status gdn_verify(float *state, const void *tape_k, const void *tape_v,
                            const float *tape_g, const float *tape_beta, int n_replay,
                            const void *q, const void *k, const void *v, const float *g,
                            const float *beta, void *o, sv_dtype o_dtype, int M, int Hk, int Hv,
                            int dk, int dv, sv_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Draft depth                                                              */
/* ---------------------------------------------------------------------- */
/* The depth with the most tokens per microsecond from measured cost curves
 * ("Speculative decoding and MTP on Apple silicon", Facts: mlx-dspark picks
 * the draft cap from the verify and drafter cost curves measured once per
 * machine; MTPLX keeps a depth only if it beats plain decoding).
 *   verify_us[K], K = 0..Kmax: host, cost of one verify pass with K+1 rows
 *     (K = 0: the plain decode step), > 0 and finite;
 *   draft_us[K]: host, cost of drafting K tokens (>= 0), or NULL for none;
 *   accept[i-1], i = 1..Kmax: host, probability that at least the first i
 *     drafts of a round are accepted (in [0, 1], non-increasing);
 *   rates_out[K]: host, receives 1 + sum_{i<=K} accept[i-1] tokens per round
 *     over verify_us[K] + draft_us[K] (tokens per microsecond), or NULL.
 * Returns the depth K with the highest rate if that rate is strictly above
 * plain decoding's (else 0; ties keep the shallower depth), or -1 on invalid
 * input.  Host code only: no GPU, no stream. */
SV_API int spec_pick_depth(const double *verify_us, const double *draft_us, const double *accept,
                           int Kmax, double *rates_out);

/* Synchronises `stream`, then reads and clears the device error word set by
 * bounded waits (SV_ERR_TIMEOUT) or candidate overflow (SV_ERR_OVERFLOW).
 * Returns SV_ERR_CUDA if the stream reports an error. */
SV_API sv_status sv_last_device_error(sv_stream_t stream);

/* Launch flags (bit set), process-wide:
 *   SV_LAUNCH_PDL: launch kernels with programmatic dependent launch, so a
 *     kernel may start while its predecessor on the stream drains.  Kernels
 *     read activations, queries, logits and workspaces and write outputs only
 *     after the predecessor has completed; the prepacked weights and the KV
 *     cache slots before kv_len-M may be read earlier, so with this flag set
 *     they must not be written by the immediately preceding kernel. */
#define SV_LAUNCH_PDL 1u
/*   SV_LAUNCH_QMM_CUDA_CORES: a measurement aid, not a faster path.
 *     qmm_small_m at M = 1 and M = 4 (72 KB-stage plans) replaces its
 *     tensor-core MMAs by fp32 FFMA on the CUDA cores (same layout, same
 *     split over CTAs, same results within the stated tolerance), so the two
 *     can be timed against each other.  Other shapes ignore it. */
#define SV_LAUNCH_QMM_CUDA_CORES 2u
/*   SV_LAUNCH_ATTN_MMA_SYNC, SV_LAUNCH_ATTN_TCGEN05: pick the kernel behind
 *     verify_attn, verify_attn_masked and verify_attn_noalloc (warp-level
 *     mma.sync tiles, or tcgen05 MMAs with tensor-memory accumulators)
 *     instead of the library's choice by query rows per KV head.  Both give
 *     the same results within the stated tolerance; MMA_SYNC wins when both
 *     are set. */
#define SV_LAUNCH_ATTN_MMA_SYNC 4u
#define SV_LAUNCH_ATTN_TCGEN05 8u
/*   SV_LAUNCH_TEST_STALL_COPY: a test aid for the bounded device waits, not for
 *     use in production.  The mma.sync attention kernel (verify_attn,
 *     verify_attn_masked and verify_attn_noalloc with SV_LAUNCH_ATTN_MMA_SYNC,
 *     or up to 16 query rows per KV head) arms its first KV copy without
 *     issuing it, and the quantised matmul (qmm_small_m, qmm8_small_m; not
 *     under its thread-block cluster plan) its first weight stage, so their
 *     waits run out after about 1.5 s of SM clocks; the call completes with
 *     an undefined output and sv_last_device_error() reports SV_ERR_TIMEOUT.
 *     The matmul's workspace stays usable for the next call.  No other
 *     kernel reads it. */
#define SV_LAUNCH_TEST_STALL_COPY 0x10000u
SV_API void sv_set_launch_flags(unsigned flags);
SV_API unsigned sv_get_launch_flags(void);

/* Number of the library's kernels launched since load (for launch-count
 * accounting; counts launches issued, including those captured into
 * graphs). */
SV_API uint64_t sv_kernel_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
