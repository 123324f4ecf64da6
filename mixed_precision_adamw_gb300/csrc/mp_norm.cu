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
// warp-shuffle tree and a fixed shared-memory pass. A block whose fp32 result
// is non-finite or below 2^-60 (possible overflow or underflow of the fp32
// squares) recomputes its share in fp64. Level 2 (norm_finalize_kernel, one
// block) adds the per-block partials in a fixed order, takes the square root
// and derives the clip scale on the device, so no host round trip is needed.
// The grid depends only on n and the SM count: results are bit-identical
// across runs.
#include <cfloat>
#include <cmath>

#include "mp_adamw.h"
#include "mp_device.cuh"
#include "mp_internal.h"

namespace mpk {
namespace {

constexpr int kNormBlocksPerSm = 4;  // 4 x 256 threads per SM, 16 B x 4 in flight each
constexpr int kUnroll = 4;           // 16-B loads in flight per thread

__device__ __forceinline__ float sumsq8(uint4 w) {
  const float a0 = bf16_lo(w.x), a1 = bf16_hi(w.x), a2 = bf16_lo(w.y), a3 = bf16_hi(w.y);
  const float a4 = bf16_lo(w.z), a5 = bf16_hi(w.z), a6 = bf16_lo(w.w), a7 = bf16_hi(w.w);
  const float s01 = __fadd_rn(__fmul_rn(a0, a0), __fmul_rn(a1, a1));
  const float s23 = __fadd_rn(__fmul_rn(a2, a2), __fmul_rn(a3, a3));
  const float s45 = __fadd_rn(__fmul_rn(a4, a4), __fmul_rn(a5, a5));
  const float s67 = __fadd_rn(__fmul_rn(a6, a6), __fmul_rn(a7, a7));
  return __fadd_rn(__fadd_rn(s01, s23), __fadd_rn(s45, s67));
}

__device__ __forceinline__ double dsumsq8(uint4 w) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  double s = 0.0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const double lo = bf16_lo(ws[j]), hi = bf16_hi(ws[j]);
    s = __dadd_rn(s, __dmul_rn(lo, lo));
    s = __dadd_rn(s, __dmul_rn(hi, hi));
  }
  return s;
}

// s + x with the rounding error of the addition accumulated in c. Both terms
// are non-negative, so max/min order them as Fast2Sum requires.
__device__ __forceinline__ void acc(float& s, float& c, float x) {
  const float t = __fadd_rn(s, x);
  const float big = fmaxf(s, x), small = fminf(s, x);
  c = __fadd_rn(c, __fadd_rn(__fsub_rn(big, t), small));
  s = t;
}

// Fixed-order block sum in fp64; every thread receives the result.
__device__ __forceinline__ double block_sum(double d, double* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) d = __dadd_rn(d, __shfl_down_sync(0xFFFFFFFFu, d, o));
  if (lane == 0) sh[warp] = d;
  __syncthreads();
  if (warp == 0) {
    double r = lane < kThreads / 32 ? sh[lane] : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r = __dadd_rn(r, __shfl_down_sync(0xFFFFFFFFu, r, o));
    if (lane == 0) sh[kThreads / 32] = r;
  }
  __syncthreads();
  const double r = sh[kThreads / 32];
  __syncthreads();  // sh may be reused by the caller
  return r;
}

// vec: grads (and copy_out) 16-B aligned, processed as 8-element vectors
// plus a scalar tail. kCopy: grads may live in page-locked host memory (read
// over the host link) and every element read is also written to copy_out, so
// the host-to-device transfer and the norm are one pass; the arithmetic and
// its order are the same as without the copy.
template <bool kCopy>
__global__ void __launch_bounds__(kThreads)
norm_partial_kernel(const uint16_t* __restrict__ grads, uint64_t n, int vec, double* __restrict__ partials,
                    uint16_t* __restrict__ copy_out) {
  __shared__ double sh[kThreads / 32 + 1];
  pdl_enter();
  const uint4* g4 = reinterpret_cast<const uint4*>(grads);
  uint4* c4 = reinterpret_cast<uint4*>(copy_out);
  const uint64_t nvec = vec ? n / 8 : 0;
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
  const uint64_t k0 = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x;

  float s = 0.0f, c = 0.0f;
  uint64_t k = k0;
  for (; k + (kUnroll - 1) * stride < nvec; k += kUnroll * stride) {
    uint4 w[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) w[u] = __ldcs(g4 + k + u * stride);
    if (kCopy) {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) c4[k + u * stride] = w[u];
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) acc(s, c, sumsq8(w[u]));
  }
  for (; k < nvec; k += stride) {
    const uint4 w = __ldcs(g4 + k);
    if (kCopy) c4[k] = w;
    acc(s, c, sumsq8(w));
  }
  for (uint64_t i = nvec * 8 + k0; i < n; i += stride) {
    const uint16_t h = grads[i];
    if (kCopy) copy_out[i] = h;
    const float x = bf16_to_f32(h);
    acc(s, c, __fmul_rn(x, x));
  }
  double S = block_sum(__dadd_rn(static_cast<double>(s), static_cast<double>(c)), sh);

  if (!(S <= DBL_MAX) || S < 0x1p-60) {  // uniform across the block: S is a broadcast value
    // Re-read this thread's own elements (from the device copy when there is
    // one: a thread always sees its own earlier writes).
    const uint4* r4 = kCopy ? reinterpret_cast<const uint4*>(copy_out) : g4;
    const uint16_t* r1 = kCopy ? copy_out : grads;
    double d = 0.0;
    for (k = k0; k < nvec; k += stride) d = __dadd_rn(d, dsumsq8(r4[k]));
    for (uint64_t i = nvec * 8 + k0; i < n; i += stride) {
      const double x = bf16_to_f32(r1[i]);
      d = __dadd_rn(d, __dmul_rn(x, x));
    }
    S = block_sum(d, sh);
  }
  if (threadIdx.x == 0) partials[blockIdx.x] = S;
}

// Advances the device step counter (one thread). Returns false, leaving the
// state untouched, when the step cannot be taken: a negative or saturated
// count, or a t beyond a bias table whose last entry is not (1, 1).
__device__ __forceinline__ bool advance_clock(const StepClock& c) {
  mp_step_state_t* st = c.state;
  const int32_t t0 = st->t;
  if (t0 < 0 || t0 == 0x7FFFFFFF) return false;
  const int32_t t = t0 + 1;
  const int64_t last = c.bias_len - 1;
  const int64_t k = (static_cast<int64_t>(t) - 1 < last) ? static_cast<int64_t>(t) - 1 : last;
  const float bc1 = c.bias[2 * k], bc2 = c.bias[2 * k + 1];
  if (static_cast<int64_t>(t) - 1 > last && !(bc1 == 1.0f && bc2 == 1.0f)) return false;
  st->t = t;
  st->seed = st->seed_base + static_cast<uint32_t>(t);
  st->bc1 = bc1;
  st->bc2 = bc2;
  return true;
}

__global__ void __launch_bounds__(kThreads)
norm_finalize_kernel(const double* __restrict__ partials, int nb, float clip,
                     float* d_norm, float* d_scale, double* d_sumsq, const StepClock clock) {
  __shared__ double sh[kThreads / 32 + 1];
  pdl_enter();
  double d = 0.0;
  for (int i = threadIdx.x; i < nb; i += kThreads) d = __dadd_rn(d, partials[i]);
  const double S = block_sum(d, sh);
  if (threadIdx.x == 0) {
    const float norm = __double2float_rn(__dsqrt_rn(S));
    float scale;
    if (!isfinite(norm)) {
      scale = __int_as_float(0x7FC00000);  // NaN: the step refuses to run
    } else {
      const float q = __fdiv_rn(clip, norm);  // norm == 0 gives +Inf -> 1
      scale = q < 1.0f ? q : 1.0f;
    }
    if (clock.state != nullptr && !advance_clock(clock)) {
      scale = __int_as_float(0x7FC00000);
      if (clock.d_status != nullptr) atomicCAS(clock.d_status, 0, MP_ERR_RANGE);
    }
    *d_norm = norm;
    *d_scale = scale;
    if (d_sumsq != nullptr) *d_sumsq = S;
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
  cudaError_t e = copy_out == nullptr
                      ? launch_pdl(norm_partial_kernel<false>, static_cast<unsigned>(nblocks), kThreads, stream,
                                   grads, n, vec ? 1 : 0, partials, copy_out)
                      : launch_pdl(norm_partial_kernel<true>, static_cast<unsigned>(nblocks), kThreads, stream,
                                   grads, n, vec ? 1 : 0, partials, copy_out);
  if (e != cudaSuccess) return e;
  return launch_pdl(norm_finalize_kernel, 1u, kThreads, stream, static_cast<const double*>(partials), nblocks,
                    clip, d_norm, d_scale, d_sumsq, c);
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
// to a kernel directly.
void* g_scratch_addr[64];

cudaError_t scratch_address(int device, double** out) {
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  void* p = g_scratch_addr[device];
  if (p == nullptr) {
    const cudaError_t e = cudaGetSymbolAddress(&p, g_norm_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[device] = p;  // racing first calls store the same address
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
