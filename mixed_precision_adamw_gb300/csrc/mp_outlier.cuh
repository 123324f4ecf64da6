// mp_outlier.cuh — the grad-norm outlier check as a device function, shared
// by its own one-thread kernel (mp_outlier.cu) and the one-launch step for
// small parameter sets (mp_small.cu).
//
// llm.c walk-through ch. 04 "Multi-GPU and mixed precision" §4: before the
// update, the train step feeds the grad norm to an outlier detector with a
// window of 128 past values and skips the update when the norm's z-score is
// above a threshold.
//
// z = (x - mean) / std over the 128 most recent finite norms (population
// standard deviation; both sums in window-slot order, fp64, one rounding per
// operation); NaN until 128 norms have been seen; the check happens before x
// joins the window; a non-finite norm never joins it.
#pragma once

#include <cstdint>

#include "mp_adamw.h"

namespace mpk {

constexpr int kWindow = 128;

struct OutlierState {
  double window[kWindow];
  unsigned long long count;  // finite norms pushed so far
};

// One check of the norm x against the window, then x joins it (if finite).
// Single thread. Returns true when the step must be skipped; stores z into
// *d_z (if given) and MP_SKIPPED_OUTLIER into *d_status (if it held 0).
__device__ __forceinline__ bool outlier_update(OutlierState* st, float norm, float z_threshold, double* d_z,
                                               int32_t* d_status) {
  const double x = static_cast<double>(norm);
  const unsigned long long count = st->count;
  double z = __longlong_as_double(0x7FF8000000000000ll);  // NaN until the window is full
  if (count >= kWindow) {
    double sum = 0.0;
#pragma unroll 1
    for (int i = 0; i < kWindow; ++i) sum = __dadd_rn(sum, st->window[i]);
    const double mean = __ddiv_rn(sum, static_cast<double>(kWindow));
    double ss = 0.0;
#pragma unroll 1
    for (int i = 0; i < kWindow; ++i) {
      const double d = __dsub_rn(st->window[i], mean);
      ss = __dadd_rn(ss, __dmul_rn(d, d));
    }
    const double sd = __dsqrt_rn(__ddiv_rn(ss, static_cast<double>(kWindow)));
    z = __ddiv_rn(__dsub_rn(x, mean), sd);
  }
  if (d_z != nullptr) *d_z = z;
  const bool skip = z_threshold > 0.0f && z > static_cast<double>(z_threshold);
  if (skip && d_status != nullptr) atomicCAS(d_status, 0, MP_SKIPPED_OUTLIER);
  if (isfinite(x)) {
    st->window[count % kWindow] = x;
    st->count = count + 1;
  }
  return skip;
}

}  // namespace mpk
