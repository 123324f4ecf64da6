// mp_internal.h — host-side interface between the C ABI (mp_api.cu) and the
// kernel launchers (mp_step.cu, mp_norm.cu, mp_sr.cu). Not installed.
#pragma once

#include <atomic>
#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

#include "mp_adamw.h"

namespace mpk {

// Decay segments: maximal runs of consecutive elements with the same decay
// flag, passed to the step kernel by value (kernel parameter space). A launch
// takes at most kSegCapLarge of them; the host splits longer tables into
// several launches.
constexpr uint32_t kSegCapSmall = 32;
constexpr uint32_t kSegCapLarge = 1024;

// Elements per step launch at most: longer ranges are split into near-equal
// launches of whole 2048-element tiles. In one launch over billions of
// elements the persistent blocks drift apart and DRAM streams slower; on
// GB300, launches of ~200M elements (1 ms) ran 1 % faster over GPT-2 1.5B and
// Llama-3-8B parameter sets than one launch, and much shorter ones lost
// time at the launch boundaries. The TMA-staged kernel agrees: the 8B set's
// update took 33.3 ms in 40 launches, 33.4 in 20 or 60, 33.5 in 10 or 80 and
// 34.2 ms in one.
constexpr uint64_t kMaxLaunchElems = uint64_t{3} << 26;  // 201,326,592

struct StepArgs {
  uint16_t* params;
  const uint16_t* grads;
  float* master;  // nullptr: no-master variant
  float* m;
  float* v;
  uint64_t n;     // elements in this launch
  uint64_t goff;  // global index of element 0 of this launch
  const float* d_scale;  // nullptr: scale 1
  int32_t* d_status;     // may be nullptr
  float lr, beta1, beta2, eps, wd, bc1, bc2;
  uint32_t seed;
  uint32_t nseg;         // segments covering [goff, goff + n)
  uint32_t first_decay;  // decay flag of segment 0; flags alternate after it
  // Vector path: elements [0, head) go one per thread and the tiles start at
  // element head, chosen so that the tiles' gradient and weight vectors
  // start on 128-B lines (a multiple of 4 below 64; 0 elsewhere).
  uint32_t head;
  // Non-null: lr, bc1, bc2 and seed are read from this device state (written
  // by the norm's finalize kernel earlier in the stream) instead of the
  // fields above.
  const mp_step_state_t* dstate;
};

// The device step counter of a replayable step (mp_optimizer_step_graph):
// the norm's finalize kernel advances state->t and writes that step's seed
// and bias corrections (bias[2(t-1)], bias[2(t-1)+1], clamped to the last
// entry) into the state for the update kernel.
struct StepClock {
  mp_step_state_t* state;  // nullptr: no device step counter
  const float* bias;
  int64_t bias_len;
  int32_t* d_status;       // may be nullptr
};

// Launches a kernel with programmatic dependent launch allowed (the kernel
// calls pdl_enter() before touching global memory).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), unsigned grid, unsigned block, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch_pdl with `smem` bytes of dynamic shared memory.
template <typename... Params, typename... Args>
cudaError_t launch_pdl_smem(void (*kernel)(Params...), unsigned grid, unsigned block, size_t smem,
                            cudaStream_t stream, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Asks the GPU to keep the largest shared-memory carve-out on SMs that run
// `kernel`. The TMA-staged step kernel needs most of an SM's shared memory.
// Measured on GB300: when the host-gradient copy (a persistent kernel beside
// the step) or the norm (just before it in the stream) ran without this
// preference, the step kernel's blocks waited for those kernels to leave the
// SMs, and a pipelined step took the copy's time plus much of the update's.
// Once per kernel (`done` belongs to that kernel) and device; a hint, so a
// failure is ignored.
template <typename... Params>
void prefer_max_shared(void (*kernel)(Params...), std::atomic<bool> (&done)[64]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  if (dev < 0 || dev >= 64 || done[dev].load(std::memory_order_relaxed)) return;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared) != cudaSuccess)
    cudaGetLastError();
  else
    done[dev].store(true, std::memory_order_relaxed);
}

struct DeviceInfo {
  int device;
  int sms;
};

cudaError_t device_info(DeviceInfo* out);

// Stores e as this thread's mp_last_cuda_error() and returns MP_ERR_CUDA.
int record_cuda_error(cudaError_t e);

// seg_end[s] = global index one past segment s; seg_end[nseg-1] == goff + n.
cudaError_t launch_adamw(const StepArgs& a, const uint64_t* seg_end, bool vec,
                         const DeviceInfo& dev, cudaStream_t stream);

int norm_blocks(uint64_t n, bool vec, const DeviceInfo& dev);
// copy_out != nullptr: grads may be page-locked host memory (device-visible
// address); the kernel also writes every gradient to copy_out (device).
// clock != nullptr: the finalize kernel also advances the device step counter.
// d_norm == nullptr (then d_scale and clock are unused): only d_sumsq is written.
cudaError_t launch_norm(const uint16_t* grads, uint64_t n, bool vec, double* partials,
                        int nblocks, float clip, float* d_norm, float* d_scale,
                        double* d_sumsq, cudaStream_t stream, uint16_t* copy_out = nullptr,
                        const StepClock* clock = nullptr);

// ZeRO-1 norm: norm and scale from `count` per-rank sums of squares, added
// in index order in fp64 (one thread).
cudaError_t launch_scale_from_sumsq(const double* parts, int count, float clip, float* d_norm, float* d_scale,
                                    double* d_total, cudaStream_t stream);

// One-launch step for small parameter sets (mp_small.cu): a cluster of
// kSmallClusterCtas CTAs runs the norm, the optional outlier check and the
// update, with results identical to the separate kernels; each CTA takes at
// most one tile and one norm block. Used by the whole-step calls when
// n <= kSmallMaxN, the update takes the vector path, the range has at most
// kSegCapSmall decay segments, the general path's norm grid has at most
// kSmallClusterCtas blocks and the GPU runs clusters of that size.
constexpr int kSmallClusterCtas = 16;
constexpr uint64_t kSmallMaxN = static_cast<uint64_t>(kSmallClusterCtas) * 2048;

// Whether the current device can launch the small step's cluster (queried
// once per device and variant).
bool small_step_available(const DeviceInfo& dev, bool master);

struct SmallArgs {
  const uint16_t* norm_src;  // gradients the norm reads (device-visible address)
  uint16_t* copy_out;        // non-null: norm_src is host memory, copied here (== StepArgs::grads)
  int32_t nb;                // norm blocks of the general path for this n
  int32_t norm_vec;          // the general path's norm takes 16-B vectors
  float clip;
  float* d_norm;
  float* d_scale;            // the same buffer as StepArgs::d_scale, written here
  StepClock clock;           // state == nullptr: t, seed, lr come from StepArgs
  void* outlier;             // nullptr: no outlier check
  float outlier_z;
  double* d_z;
};

cudaError_t launch_small_step(const StepArgs& a, const SmallArgs& s, const uint64_t* seg_end,
                              cudaStream_t stream);

// Outlier check of the grad norm (mp_outlier.cu): d_state holds the window.
cudaError_t launch_outlier_check(void* d_state, const float* d_norm, float z_threshold, float* d_scale,
                                 double* d_z, int32_t* d_status, cudaStream_t stream);

cudaError_t launch_sr(uint16_t* out, const float* in, uint64_t goff, uint64_t n,
                      uint32_t seed, bool vec, const DeviceInfo& dev, cudaStream_t stream);

cudaError_t launch_sr_fp16(uint16_t* out, const float* in, uint64_t goff, uint64_t n, uint32_t seed, bool vec,
                           const DeviceInfo& dev, cudaStream_t stream);

cudaError_t launch_accumulate_sr(uint16_t* acc, const float* delta, uint64_t goff, uint64_t n, uint32_t seed,
                                 bool vec, const DeviceInfo& dev, cudaStream_t stream);

cudaError_t launch_noise(uint32_t* out, uint64_t first, uint64_t n, uint32_t seed,
                         const DeviceInfo& dev, cudaStream_t stream);

}  // namespace mpk
