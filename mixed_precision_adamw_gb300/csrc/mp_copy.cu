// mp_copy.cu — host-to-device copies by the SMs, for gradients that arrive in
// page-locked host memory.
//
// llm.c walk-through ch. 04 "Multi-GPU and mixed precision" §3.3 hides
// transfers behind compute on a second stream. Here the transfer is the next
// step's gradients crossing the host link while the current step's update
// streams through HBM. Alone, a copy engine and SM loads both move pinned
// host memory at the link's ~210 GB/s on GB300; but in some runs of pipelined
// steps on some GB300 hosts, the copy engine's 16 GB took ~175 ms where SM
// loads of the same buffer in the same process took ~92 ms. One block of 256
// threads per SM, at a few dozen registers and no shared memory, fits beside
// the update kernel's block (608 threads, 129 KB of shared memory on long
// ranges; three blocks of 256 threads on short ones), so the copy runs
// concurrently with the update rather than after it. Two or four blocks per
// SM copy as fast alone but serialised with the update in a pipelined step.
#include <cstdint>

#include "mp_adamw.h"
#include "mp_device.cuh"
#include "mp_internal.h"

namespace mpk {
namespace {

constexpr int kCopyUnroll = 4;  // 16-B loads in flight per thread

// dst[i] = src[i] for n 16-B vectors, then the tail bytes one by one.
__global__ void __launch_bounds__(kThreads)
copy_from_host_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, uint64_t nvec,
                      uint8_t* __restrict__ dst_tail, const uint8_t* __restrict__ src_tail, uint64_t ntail) {
  pdl_enter();
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
  uint64_t i = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x;
  for (; i + (kCopyUnroll - 1) * stride < nvec; i += kCopyUnroll * stride) {
    uint4 w[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) w[u] = src[i + u * stride];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) dst[i + u * stride] = w[u];
  }
  for (; i < nvec; i += stride) dst[i] = src[i];
  for (uint64_t j = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x; j < ntail; j += stride)
    dst_tail[j] = src_tail[j];
}

// Byte by byte, for buffers that are not both 16-B aligned.
__global__ void __launch_bounds__(kThreads)
copy_from_host_bytes_kernel(uint8_t* __restrict__ dst, const uint8_t* __restrict__ src, uint64_t n) {
  pdl_enter();
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n; i += stride) dst[i] = src[i];
}

}  // namespace
}  // namespace mpk

extern "C" int mp_copy_from_host(void* dst, const void* host_src, uint64_t bytes, int32_t blocks_per_sm,
                                 void* stream) {
  if (bytes == 0) return MP_OK;
  if (dst == nullptr || host_src == nullptr) return MP_ERR_NULL;
  if (blocks_per_sm < 1 || blocks_per_sm > 32 || bytes > (uint64_t{1} << 62)) return MP_ERR_RANGE;
  // The source must be page-locked host memory with a device-visible address.
  cudaPointerAttributes attr{};
  cudaError_t e = cudaPointerGetAttributes(&attr, host_src);
  if (e != cudaSuccess) {
    cudaGetLastError();  // clear the non-sticky error this query may leave
    return MP_ERR_ACCESS;
  }
  if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) return MP_ERR_ACCESS;
  const uint8_t* src = static_cast<const uint8_t*>(attr.devicePointer);
  mpk::DeviceInfo dev;
  e = mpk::device_info(&dev);
  if (e != cudaSuccess) return mpk::record_cuda_error(e);
  const unsigned grid = static_cast<unsigned>(dev.sms * blocks_per_sm);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* d = static_cast<uint8_t*>(dst);
  static std::atomic<bool> carve_vec[64], carve_bytes[64];
  if (reinterpret_cast<uintptr_t>(src) % 16 == 0 && reinterpret_cast<uintptr_t>(d) % 16 == 0) {
    mpk::prefer_max_shared(mpk::copy_from_host_kernel, carve_vec);
    const uint64_t nvec = bytes / 16, done = nvec * 16;
    e = mpk::launch_pdl(mpk::copy_from_host_kernel, grid, mpk::kThreads, s, reinterpret_cast<uint4*>(d),
                        reinterpret_cast<const uint4*>(src), nvec, d + done, src + done, bytes - done);
  } else {
    mpk::prefer_max_shared(mpk::copy_from_host_bytes_kernel, carve_bytes);
    e = mpk::launch_pdl(mpk::copy_from_host_bytes_kernel, grid, mpk::kThreads, s, d, src, bytes);
  }
  if (e != cudaSuccess) return mpk::record_cuda_error(e);
  return MP_OK;
}
