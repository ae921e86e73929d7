// accept_common.cuh -- pieces shared by the two paths of spec_accept: the
// candidate-list path (accept.cu: top-k of at most 1024, or temperature 0) and
// the whole-vocabulary path (accept_whole.cu: every other setting).
#pragma once

#include "common.cuh"

namespace sv {
namespace acc {

constexpr int MAX_K = 32;       // drafts per round
constexpr int MAX_TOPK = 1024;  // largest top-k of the candidate-list path
constexpr int MAX_CHUNKS = 64;  // CTAs per logits row
constexpr int MIN_CHUNK = 2048; // logits per CTA at least

// Order-preserving integer image of a logit: a < b as floats iff
// fkey(a) < fkey(b) as unsigned integers (NaN excluded; -0 and +0 equal).
__device__ __forceinline__ uint32_t fkey(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float keyf(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Streaming load (evict first): the row is read once.
template <typename T>
__device__ __forceinline__ float load_logit(const T *p, long long i);
template <>
__device__ __forceinline__ float load_logit<float>(const float *p, long long i) {
  return __ldcs(p + i);
}
template <>
__device__ __forceinline__ float load_logit<__nv_bfloat16>(const __nv_bfloat16 *p, long long i) {
  const unsigned short b = __ldcs(reinterpret_cast<const unsigned short *>(p) + i);
  return __uint_as_float((uint32_t)b << 16);
}

// Cached load: the row is read again by a later pass of the same call.
template <typename T>
__device__ __forceinline__ float load_logit_keep(const T *p, long long i);
template <>
__device__ __forceinline__ float load_logit_keep<float>(const float *p, long long i) {
  return __ldg(p + i);
}
template <>
__device__ __forceinline__ float load_logit_keep<__nv_bfloat16>(const __nv_bfloat16 *p, long long i) {
  const unsigned short b = __ldg(reinterpret_cast<const unsigned short *>(p) + i);
  return __uint_as_float((uint32_t)b << 16);
}

// Row j of round r: j <= K is target row j, else draft row j-K-1.
template <typename T>
__device__ __forceinline__ const T *row_ptr(const T *tgt, const T *drf, int r, int j, int K, int V) {
  return j <= K ? tgt + ((size_t)r * (K + 1) + j) * V : drf + ((size_t)r * K + (j - K - 1)) * V;
}

// Chunks per row: enough CTAs to cover the SMs twice when there are few rows,
// at least MIN_CHUNK logits each; and (k > 0, candidate-list path) few enough
// that the chunks' top-k lists fit the merging CTA's buffer (`buf` keys)
// together.  With k = 0 the result is the most chunks any k could use
// (workspace sizing).
__host__ __device__ inline int chunks_per_row(long long rows, int V, int sms, int k = 0,
                                              int buf = 0) {
  if (sms <= 0) return 1;
  long long c = (2LL * sms + rows - 1) / rows;
  c = c < 1 ? 1 : c;
  c = c > MAX_CHUNKS ? MAX_CHUNKS : c;
  const long long cmax = V / MIN_CHUNK;
  if (c > cmax) c = cmax < 1 ? 1 : cmax;
  if (k > 0 && c > buf / (2LL * k)) c = buf / (2LL * k) < 1 ? 1 : buf / (2LL * k);
  return (int)c;
}

// The whole-vocabulary path (accept_whole.cu).
struct WholeArgs {
  const void *tgt, *drf;
  int bf16;
  const int32_t *drafts;
  const float *u;
  int32_t *out_tok, *out_n;
  int R, K, V;
  float temperature;  // > 0
  int top_k;          // 0 = off (callers pass 0 for top_k >= V)
  float top_p;        // in (0, 1]; 1 = off
  void *workspace;    // the whole path's region, zeroed once
  size_t ws_bytes;
};
size_t whole_workspace_bytes(int R, int K, int V);
sv_status whole_launch(const WholeArgs &a, cudaStream_t s);

}  // namespace acc
}  // namespace sv
