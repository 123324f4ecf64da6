// mp_outlier.cu — grad-norm outlier check on the device.
//
// llm.c walk-through ch. 04 "Multi-GPU and mixed precision" §4: before the
// update, the train step feeds the grad norm to an outlier detector with a
// window of 128 past values and skips the update when the norm's z-score is
// above a threshold. Here the detector runs as a one-thread kernel between
// mp_grad_norm and mp_adamw_step, reading the norm and writing the clip scale
// in device memory, so the step needs no host round trip: a skipped step is
// a NaN scale (the step kernel then writes nothing) plus a status code. The
// check itself (mp_outlier.cuh) is shared with the one-launch small step.
#include <cmath>

#include "mp_adamw.h"
#include "mp_device.cuh"
#include "mp_internal.h"
#include "mp_outlier.cuh"

namespace mpk {
namespace {

__global__ void outlier_check_kernel(OutlierState* st, const float* d_norm, float z_threshold, float* d_scale,
                                     double* d_z, int32_t* d_status) {
  pdl_enter();
  if (outlier_update(st, *d_norm, z_threshold, d_z, d_status)) *d_scale = __int_as_float(0x7FC00000);
}

}  // namespace

cudaError_t launch_outlier_check(void* d_state, const float* d_norm, float z_threshold, float* d_scale,
                                 double* d_z, int32_t* d_status, cudaStream_t stream) {
  return launch_pdl(outlier_check_kernel, 1u, 1u, stream, static_cast<OutlierState*>(d_state), d_norm,
                    z_threshold, d_scale, d_z, d_status);
}

}  // namespace mpk

extern "C" size_t mp_outlier_state_bytes(void) { return sizeof(mpk::OutlierState); }

extern "C" int mp_outlier_reset(void* d_state, void* stream) {
  if (d_state == nullptr) return MP_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(d_state) % 8) return MP_ERR_ALIGN;
  const cudaError_t e =
      cudaMemsetAsync(d_state, 0, sizeof(mpk::OutlierState), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return mpk::record_cuda_error(e);
  return MP_OK;
}

extern "C" int mp_outlier_check(void* d_state, const float* d_norm, float z_threshold, float* d_scale,
                                double* d_z, int32_t* d_status, void* stream) {
  if (d_state == nullptr || d_norm == nullptr || d_scale == nullptr) return MP_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(d_state) % 8 || reinterpret_cast<uintptr_t>(d_norm) % 4 ||
      reinterpret_cast<uintptr_t>(d_scale) % 4 || reinterpret_cast<uintptr_t>(d_z) % 8 ||
      reinterpret_cast<uintptr_t>(d_status) % 4)
    return MP_ERR_ALIGN;
  const cudaError_t e = mpk::launch_outlier_check(d_state, d_norm, z_threshold, d_scale, d_z, d_status,
                                                   static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return mpk::record_cuda_error(e);
  return MP_OK;
}
