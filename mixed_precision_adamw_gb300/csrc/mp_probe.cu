// mp_probe.cu — compute-free stream probes for the benchmark (libmpprobe.so).
//
// Measurement only: not part of the optimizer's ABI, loaded by bench.py alone.
// They answer one question: how fast can kernels on the SMs move exactly the
// memory streams of the optimizer step on this GPU, with no arithmetic in
// between? The step reads a bf16 gradient and fp32 master, m, v and writes
// fp32 master, m, v and a bf16 weight (28 B per parameter, half read, half
// written). The probes use the step kernel's tiling (thread t takes the
// 4-element groups at tile offsets 4t and 4t + 1024 of a 2048-element tile,
// 16-B fp32 and 8-B bf16 vectors, streaming cache hints) and its grid
// (persistent blocks, a given number per SM), and write back what they read.
// A plain 16-B vector copy of the same bytes is the second probe. Their
// throughput is the practical ceiling for the step kernel on the SMs; the
// copy engines (cudaMemcpyAsync) are measured separately by the benchmark.
#include <cstdint>

#include <cuda_runtime.h>

namespace {

constexpr int kThreads = 256;
constexpr int kTile = 2048;

// The step's five streams, values carried through unchanged: the "update"
// writes master, m and v back and packs the gradient's bits into the weight.
__global__ void __launch_bounds__(kThreads)
step_streams_probe(uint16_t* __restrict__ params, const uint16_t* __restrict__ grads, float* __restrict__ master,
                   float* __restrict__ m, float* __restrict__ v, uint64_t n) {
  const uint64_t ntiles = n / kTile;
  for (uint64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const uint64_t e0 = tile * kTile + threadIdx.x * 4;
    const uint64_t e1 = e0 + kThreads * 4;
    const uint2 g0 = __ldcs(reinterpret_cast<const uint2*>(grads + e0));
    const uint2 g1 = __ldcs(reinterpret_cast<const uint2*>(grads + e1));
    const float4 m0 = __ldcs(reinterpret_cast<const float4*>(m + e0));
    const float4 m1 = __ldcs(reinterpret_cast<const float4*>(m + e1));
    const float4 v0 = __ldcs(reinterpret_cast<const float4*>(v + e0));
    const float4 v1 = __ldcs(reinterpret_cast<const float4*>(v + e1));
    const float4 w0 = __ldcs(reinterpret_cast<const float4*>(master + e0));
    const float4 w1 = __ldcs(reinterpret_cast<const float4*>(master + e1));
    __stcs(reinterpret_cast<float4*>(m + e0), m0);
    __stcs(reinterpret_cast<float4*>(m + e1), m1);
    __stcs(reinterpret_cast<float4*>(v + e0), v0);
    __stcs(reinterpret_cast<float4*>(v + e1), v1);
    __stcs(reinterpret_cast<float4*>(master + e0), w0);
    __stcs(reinterpret_cast<float4*>(master + e1), w1);
    __stcs(reinterpret_cast<uint2*>(params + e0), g0);
    __stcs(reinterpret_cast<uint2*>(params + e1), g1);
  }
}

// dst[i] = src[i] over n 16-B vectors.
__global__ void __launch_bounds__(kThreads)
copy_probe(uint4* __restrict__ dst, const uint4* __restrict__ src, uint64_t n) {
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n; i += stride)
    __stcs(dst + i, __ldcs(src + i));
}

int grid(int blocks_per_sm) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms * blocks_per_sm;
}

}  // namespace

extern "C" {

// The step's streams over n parameters (n a multiple of 2048; params and
// grads 8-B aligned, master, m, v 16-B aligned; device pointers), with
// blocks_per_sm persistent blocks per SM. Returns a cudaError_t.
int mp_probe_step_streams(uint16_t* params, const uint16_t* grads, float* master, float* m, float* v, uint64_t n,
                          int blocks_per_sm, void* stream) {
  const int g = grid(blocks_per_sm);
  if (g <= 0 || n % kTile) return static_cast<int>(cudaErrorInvalidValue);
  step_streams_probe<<<g, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(params, grads, master, m, v, n);
  return static_cast<int>(cudaGetLastError());
}

// A 16-B vector copy of n_vec16 vectors (both pointers 16-B aligned).
int mp_probe_copy(void* dst, const void* src, uint64_t n_vec16, int blocks_per_sm, void* stream) {
  const int g = grid(blocks_per_sm);
  if (g <= 0) return static_cast<int>(cudaErrorInvalidValue);
  copy_probe<<<g, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint4*>(dst),
                                                                    static_cast<const uint4*>(src), n_vec16);
  return static_cast<int>(cudaGetLastError());
}

}  // extern "C"
