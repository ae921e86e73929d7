// depth.cu -- draft depth from measured cost curves (host code).
//
// "Speculative decoding and MTP on Apple silicon", Facts: mlx-dspark measures
// the verify and drafter cost curves on the user's machine once and picks the
// draft cap from them (different chips pick different caps); MTPLX keeps a
// depth only if it beats plain decoding.  With the verify cost table that
// the benchmark measures per context (verify_attn and qmm_small_m at M rows),
// this picks the depth that yields the most tokens per microsecond.
#include <cmath>

#include "common.cuh"

extern "C" {

int spec_pick_depth(const double *verify_us, const double *draft_us, const double *accept, int Kmax,
                    double *rates_out) {
  if (Kmax < 0 || !verify_us || (Kmax > 0 && !accept)) return -1;
  for (int K = 0; K <= Kmax; ++K) {
    const double d = draft_us ? draft_us[K] : 0.0;
    if (!(verify_us[K] > 0.0) || !std::isfinite(verify_us[K])) return -1;
    if (!(d >= 0.0) || !std::isfinite(d)) return -1;
  }
  for (int i = 0; i < Kmax; ++i) {
    if (!(accept[i] >= 0.0 && accept[i] <= 1.0)) return -1;
    if (i > 0 && accept[i] > accept[i - 1]) return -1;  // at least i+1 accepted <= at least i
  }
  // expected tokens of a round at depth K: the accepted drafts plus the
  // one token every round emits (correction or bonus)
  double tokens = 1.0;
  int best = 0;
  double best_rate = 0.0;
  for (int K = 0; K <= Kmax; ++K) {
    if (K > 0) tokens += accept[K - 1];
    const double rate = tokens / (verify_us[K] + (draft_us ? draft_us[K] : 0.0));
    if (rates_out) rates_out[K] = rate;
    if (K == 0 || rate > best_rate) {  // strictly better: ties keep the shallower depth
      best = K;
      best_rate = rate;
    }
  }
  return best;
}

}  // extern "C"
