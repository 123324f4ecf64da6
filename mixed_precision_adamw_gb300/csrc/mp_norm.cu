// mp_norm.cu — deterministic global gradient norm and clip scale.
//
// llm.c walk-through ch. 04 "Multi-GPU and mixed precision" §4: the train
// step computes the global norm of all gradients with a two-level reduction
// kernel, then grad_scale = min(1, 1.0 / grad_norm).
//
// Level 1 (norm_partial_kernel, persistent grid): each thread squares its
// bf16 gradients in fp32 (exact for |g| in [2^-63, 2^64)), adds each 8-element
// vector as a pairwise tree and accumulates the vector sums with Fast2Sum
// compensation; the threads of a block are reduced in fp64 by a fixed
// warp-shuffle tree and a fixed shared-memory pass. For long aligned device
// gradients norm_partial_tma_kernel does the same additions in the same
// order on vectors that the TMA engine stages in shared memory. A block whose fp32 result
// is non-finite or below 2^-60 (possible overflow or underflow of the fp32
// squares) recomputes its share in fp64. Level 2 (norm_finalize_kernel, one
// block) adds the per-block partials in a fixed order, takes the square root
// and derives the clip scale on the device, so no host round trip is needed.
// The grid and the element mapping depend only on n, the SM count and whether
// the gradients are 16-B aligned (8-element vectors) or not (single
// elements): results are bit-identical across runs.
#include <atomic>
#include <cmath>

#include "mp_adamw.h"
#include "mp_device.cuh"
#include "mp_internal.h"
#include "mp_norm.cuh"
#include "mp_tma.cuh"

namespace mpk {
namespace {

constexpr int kNormBlocksPerSm = 4;  // 4 x 256 threads per SM, 16 B x 4 in flight each

// Level 1: one norm block per CTA (mp_norm.cuh has the arithmetic).
template <bool kCopy>
__global__ void __launch_bounds__(kThreads)
norm_partial_kernel(const uint16_t* __restrict__ grads, uint64_t n, int vec, double* __restrict__ partials,
                    uint16_t* __restrict__ copy_out) {
  __shared__ double sh[kThreads / 32 + 1];
  pdl_enter();
  const double S = norm_block_partial<kCopy>(grads, n, vec, copy_out, blockIdx.x, gridDim.x, sh);
  if (threadIdx.x == 0) partials[blockIdx.x] = S;
}

// Level 1 with the gradients staged through shared memory by the TMA engine,
// for 16-B aligned device gradients: the element mapping and the order of
// every addition are norm_partial_kernel's, so each partial has the same bits.
// Launched only where norm_map gives each block a contiguous run of 4 KB
// pieces (256 vectors each). Thread 0 has groups of kNormPiecesPerStage
// consecutive pieces loaded, one bulk copy per group, into a ring of
// kNormTmaStages stages while the block adds the pieces of an earlier group
// in order (thread t the vector t of each); a stage is loaded again once
// every warp has read it (an mbarrier per stage each way).
// Measured on GB300 (Llama-3-8B gradients, 16 GB): 4 pieces x 3 stages
// 2.15-2.18 ms; 8 x 2 3.03. With the blocks' pieces interleaved (4 KB bulk
// copies, 1 to 8 per group) the best shape took 2.46 ms (4 x 3; 3 x 4 2.50;
// 6 x 2 2.65; 2 x 6 3.09; 1 x 8 2.90), and the register kernel 2.55 ms in
// the same shared-memory configuration. The loads do not pass through L1, so
// the kernel keeps its rate with most of the SM's memory as shared memory,
// where the TMA-staged step kernel must run beside or after it (with it the
// norm -> update boundary of a step costs nothing measurable; with the
// register kernel it cost 0.3 ms). Every wait gives up after one second; a
// block that gave up writes a NaN partial, so the norm and scale come out NaN
// and the step refuses to run.
constexpr uint32_t kNormTmaStages = 3;
constexpr uint32_t kNormPiecesPerStage = 4;
constexpr uint32_t kNormPieceBytes = kThreads * 16;
constexpr uint32_t kNormStageBytes = kNormPiecesPerStage * kNormPieceBytes;
constexpr size_t kNormTmaSmem = kNormTmaStages * kNormStageBytes + 16 * kNormTmaStages;

__global__ void __launch_bounds__(kThreads)
norm_partial_tma_kernel(const uint16_t* __restrict__ grads, uint64_t n, double* __restrict__ partials) {
  __shared__ double sh[kThreads / 32 + 1];
  __shared__ int gave_up;
  extern __shared__ __align__(128) uint8_t ring[];
  pdl_enter();
  constexpr uint32_t S = kNormTmaStages, G = kNormPiecesPerStage;
  const uint32_t base = smem_u32(ring), full = base + S * kNormStageBytes, done = full + 8 * S;
  const uint64_t nvec = n / 8;
  const NormMap map = norm_map(nvec, blockIdx.x, gridDim.x);  // contiguous: the launch ensures it
  const uint64_t first = map.first, last = map.last;
  const uint64_t pieces = (last - first + kThreads - 1) / kThreads;  // 256-vector pieces
  const uint64_t groups = (pieces + G - 1) / G;  // one bulk copy: pieces G*q .. G*q + G - 1
  if (threadIdx.x == 0) {
    gave_up = 0;
    for (uint32_t i = 0; i < S; ++i) {
      mbar_init(full + 8 * i, 1);
      mbar_init(done + 8 * i, kThreads / 32);
    }
    mbar_init_fence();
  }
  __syncthreads();
  const uint4* g4 = reinterpret_cast<const uint4*>(grads);
  uint64_t policy = 0, issued = 0;
  auto load = [&](uint64_t q) {
    const uint32_t st = static_cast<uint32_t>(q % S);
    const uint64_t v0 = first + q * G * kThreads;
    const uint64_t v1 = v0 + G * kThreads < last ? v0 + G * kThreads : last;
    const uint32_t bytes = static_cast<uint32_t>((v1 - v0) * 16);
    mbar_expect_tx(full + 8 * st, bytes);
    bulk_load(base + st * kNormStageBytes, g4 + v0, bytes, full + 8 * st, policy);
  };
  bool producing = threadIdx.x == 0;
  if (producing) {
    policy = l2_evict_first();
    for (; issued < groups && issued + 1 < S; ++issued) load(issued);
  }
  float s = 0.0f, c = 0.0f;
  uint64_t q = 0;
  for (; q < groups; ++q) {
    const uint32_t st = static_cast<uint32_t>(q % S);
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(full + 8 * st, static_cast<uint32_t>((q / S) & 1)))) {
      if ((threadIdx.x & 31) == 0) atomicExch(&gave_up, 1);
      break;
    }
    const uint8_t* sp = ring + st * kNormStageBytes + 16u * threadIdx.x;
#pragma unroll
    for (uint32_t g = 0; g < G; ++g) {
      const uint64_t p = q * G + g;
      if (p < pieces && first + p * kThreads + threadIdx.x < last)
        acc(s, c, sumsq8(*reinterpret_cast<const uint4*>(sp + g * kNormPieceBytes)));
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(done + 8 * st);
    if (producing && issued < groups) {
      // group `issued` (q + S - 1) goes into the stage that group q - 1 used
      if (q >= 1 && !mbar_wait(done + 8 * ((q - 1) % S), static_cast<uint32_t>(((q - 1) / S) & 1))) {
        atomicExch(&gave_up, 1);
        producing = false;
      } else {
        load(issued++);
      }
    }
  }
  if (threadIdx.x == 0)  // loads this thread issued and did not see land: bounded waits
    for (uint64_t p = q; p < issued; ++p)
      mbar_wait(full + 8 * static_cast<uint32_t>(p % S), static_cast<uint32_t>((p / S) & 1));
  const double P = norm_block_finish<false>(grads, n, 1, nullptr, blockIdx.x, gridDim.x, sh, s, c);
  if (threadIdx.x == 0) partials[blockIdx.x] = gave_up ? __longlong_as_double(0x7FF8000000000000ll) : P;
}

__global__ void __launch_bounds__(kThreads)
norm_finalize_kernel(const double* __restrict__ partials, int nb, float clip,
                     float* d_norm, float* d_scale, double* d_sumsq, const StepClock clock) {
  __shared__ double sh[kThreads / 32 + 1];
  pdl_enter();
  const double S = norm_total([partials](int i) { return partials[i]; }, nb, sh);
  if (threadIdx.x == 0) {
    if (d_norm != nullptr) {  // null: the sum of squares alone (mp_grad_sumsq)
      float norm, scale;
      norm_and_scale(S, clip, norm, scale);
      if (clock.state != nullptr && !advance_clock(clock)) {
        scale = __int_as_float(0x7FC00000);
        if (clock.d_status != nullptr) atomicCAS(clock.d_status, 0, MP_ERR_RANGE);
      }
      *d_norm = norm;
      *d_scale = scale;
    }
    if (d_sumsq != nullptr) *d_sumsq = S;
  }
}

// The norm and clip scale from `count` sums of squares (one per ZeRO-1
// rank), added in index order in fp64 by one thread.
__global__ void __launch_bounds__(32)
scale_from_sumsq_kernel(const double* __restrict__ parts, int count, float clip, float* d_norm, float* d_scale,
                        double* d_total) {
  pdl_enter();
  if (threadIdx.x == 0) {
    double S = 0.0;
    for (int r = 0; r < count; ++r) S = __dadd_rn(S, parts[r]);
    float norm, scale;
    norm_and_scale(S, clip, norm, scale);
    *d_norm = norm;
    *d_scale = scale;
    if (d_total != nullptr) *d_total = S;
  }
}

}  // namespace

int norm_blocks(uint64_t n, bool vec, const DeviceInfo& dev) {
  const uint64_t items = vec ? (n / 8 > 0 ? n / 8 : n) : n;
  uint64_t blocks = (items + kThreads - 1) / kThreads;
  const uint64_t cap = static_cast<uint64_t>(dev.sms) * kNormBlocksPerSm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<int>(blocks);
}

cudaError_t launch_norm(const uint16_t* grads, uint64_t n, bool vec, double* partials, int nblocks,
                        float clip, float* d_norm, float* d_scale, double* d_sumsq, cudaStream_t stream,
                        uint16_t* copy_out, const StepClock* clock) {
  const StepClock c = clock != nullptr ? *clock : StepClock{nullptr, nullptr, 0, nullptr};
  // Aligned device gradients with at least two pieces per block take the
  // TMA-staged kernel (the same partials, bit for bit), which keeps its rate
  // in the large shared-memory configuration the TMA-staged step kernel
  // needs. The other kernels here ask for that configuration too, so that the
  // step kernel can share SMs with them. Measured on GB300: without it a
  // pipelined 2B-param step took 24-25 ms instead of 19.5 ms; with it (any
  // explicit carve-out from 25 % up) the register partial kernel runs alone
  // about 15 % slower.
  static std::atomic<bool> carve_plain[64], carve_copy[64], carve_finalize[64];
  prefer_max_shared(norm_finalize_kernel, carve_finalize);
  const uint64_t stride = static_cast<uint64_t>(nblocks) * kThreads;
  if (vec && copy_out == nullptr && n / 8 >= 2 * stride) {
    static std::atomic<bool> smem_set[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !smem_set[dev].load(std::memory_order_relaxed)) {
      e = cudaFuncSetAttribute(norm_partial_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kNormTmaSmem));
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) smem_set[dev].store(true, std::memory_order_relaxed);
    }
    e = launch_pdl_smem(norm_partial_tma_kernel, static_cast<unsigned>(nblocks), kThreads,
                        kNormTmaSmem, stream, grads, n, partials);
    if (e != cudaSuccess) return e;
    return launch_pdl(norm_finalize_kernel, 1u, kThreads, stream, static_cast<const double*>(partials), nblocks,
                      clip, d_norm, d_scale, d_sumsq, c);
  }
  if (copy_out == nullptr) prefer_max_shared(norm_partial_kernel<false>, carve_plain);
  else prefer_max_shared(norm_partial_kernel<true>, carve_copy);
  cudaError_t e = copy_out == nullptr
                      ? launch_pdl(norm_partial_kernel<false>, static_cast<unsigned>(nblocks), kThreads, stream,
                                   grads, n, vec ? 1 : 0, partials, copy_out)
                      : launch_pdl(norm_partial_kernel<true>, static_cast<unsigned>(nblocks), kThreads, stream,
                                   grads, n, vec ? 1 : 0, partials, copy_out);
  if (e != cudaSuccess) return e;
  return launch_pdl(norm_finalize_kernel, 1u, kThreads, stream, static_cast<const double*>(partials), nblocks,
                    clip, d_norm, d_scale, d_sumsq, c);
}

cudaError_t launch_scale_from_sumsq(const double* parts, int count, float clip, float* d_norm, float* d_scale,
                                    double* d_total, cudaStream_t stream) {
  return launch_pdl(scale_from_sumsq_kernel, 1u, 32u, stream, parts, count, clip, d_norm, d_scale, d_total);
}

}  // namespace mpk

// ---------------------------------------------------------------------------
// mp_grad_norm_noalloc: the same two kernels, with the per-block partial sums
// kept in a scratch array that this library defines itself, so the caller
// passes no workspace and nothing is allocated on any call.
// ---------------------------------------------------------------------------
namespace {

// Room for 4096 fp64 partials (32 KB). Every GPU that loads the library keeps
// this array until the process exits. A call needs one slot per norm block:
// at most 4 x SMs (608 on a 152-SM GB300).
constexpr int kNoAllocMaxPartials = 4096;
static __device__ __align__(256) double g_norm_scratch[kNoAllocMaxPartials];

// Device address of g_norm_scratch, looked up once per device (with that
// device current) on the first call made on it. In host code the array's name
// is only a host-side stand-in, never a device address, so it is not passed
// to a kernel directly. The cache is keyed by device ordinal and assumes that
// device's primary context for the life of the process (no cudaDeviceReset).
// Ordinals past the cache are looked up on every call.
constexpr int kAddrCache = 64;
std::atomic<void*> g_scratch_addr[kAddrCache];

cudaError_t scratch_address(int device, double** out) {
  const bool cached = device >= 0 && device < kAddrCache;
  void* p = cached ? g_scratch_addr[device].load(std::memory_order_relaxed) : nullptr;
  if (p == nullptr) {
    const cudaError_t e = cudaGetSymbolAddress(&p, g_norm_scratch);
    if (e != cudaSuccess) return e;
    // racing first calls on one device store the same address
    if (cached) g_scratch_addr[device].store(p, std::memory_order_relaxed);
  }
  *out = static_cast<double*>(p);
  return cudaSuccess;
}

}  // namespace

// For callers that cannot allocate device memory (a framework that owns all
// of it and passes in only the tensors, or a loop that must not take the
// device-wide synchronisation of cudaMalloc/cudaFree): the caller passes the
// inputs and outputs, and the partial sums go to g_norm_scratch. No call
// allocates anything. Overlapping calls on one device race on the scratch.
extern "C" int mp_grad_norm_noalloc(const uint16_t* grads, uint64_t n, float clip, float* d_norm,
                                    float* d_scale, double* d_sumsq, void* stream) {
  if ((n != 0 && grads == nullptr) || d_norm == nullptr || d_scale == nullptr) return MP_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(grads) % 2 || reinterpret_cast<uintptr_t>(d_norm) % 4 ||
      reinterpret_cast<uintptr_t>(d_scale) % 4 || reinterpret_cast<uintptr_t>(d_sumsq) % 8)
    return MP_ERR_ALIGN;
  if (!(clip > 0.0f) || !isfinite(clip) || n > (1ull << 62)) return MP_ERR_RANGE;
  mpk::DeviceInfo dev;
  cudaError_t e = mpk::device_info(&dev);
  if (e != cudaSuccess) return mpk::record_cuda_error(e);
  const bool vec = reinterpret_cast<uintptr_t>(grads) % 16 == 0;
  const int nb = mpk::norm_blocks(n, vec, dev);
  if (nb > kNoAllocMaxPartials) return MP_ERR_WORKSPACE;  // a GPU with more than 1024 SMs
  double* scratch = nullptr;
  e = scratch_address(dev.device, &scratch);
  if (e == cudaSuccess)
    e = mpk::launch_norm(grads, n, vec, scratch, nb, clip, d_norm, d_scale, d_sumsq,
                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return mpk::record_cuda_error(e);
  return MP_OK;
}
