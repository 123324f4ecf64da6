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
//
// The third and fourth probes move the same streams through shared memory
// with the TMA engine's 1D bulk copies instead of register loads: one thread
// per block issues, per tile (2048 elements: 28 KB, or a given multiple of
// 64), four bulk loads (gradient, master, m, v) that complete on a stage's
// mbarrier, then four bulk
// stores from the staged tile (master, m and v back, the gradient's bits into
// the weight), with several stages in flight per block; and a plain bulk
// copy in 28 KB tiles. Every wait on an mbarrier gives up after one second
// (it then sets an error word and still waits, bounded, for its copies).
#include <cstdint>

#include <cuda_runtime.h>

#include "mp_tma.cuh"

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

// ---- TMA bulk-copy probes ---------------------------------------------------
constexpr int kBulkMaxStreams = 4;
constexpr int kBulkMaxStages = 8;

struct BulkStreams {
  const uint8_t* load[kBulkMaxStreams];  // tile t of stream i starts at load[i] + t * load_bytes[i]
  uint8_t* store[kBulkMaxStreams];
  uint32_t load_bytes[kBulkMaxStreams];   // per tile, multiples of 16
  uint32_t store_bytes[kBulkMaxStreams];
  uint32_t store_from[kBulkMaxStreams];   // byte offset, in a stage, of the staged data each store writes
  int32_t nload, nstore;
  uint32_t stage_bytes;  // sum of load_bytes, a multiple of 128
  int32_t stages;        // 2 .. kBulkMaxStages
  int32_t hint;          // 1: L2 evict-first policy on every copy
  uint32_t extra_tx;     // bytes a stage's barrier expects beyond its loads (0; > 0 only to test give-up)
};

__global__ void __launch_bounds__(32)
bulk_streams_probe(const __grid_constant__ BulkStreams s, uint64_t ntiles, uint32_t* __restrict__ err) {
  if (threadIdx.x != 0) return;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  const uint32_t bars = base + static_cast<uint32_t>(s.stages) * s.stage_bytes;
  const uint32_t S = static_cast<uint32_t>(s.stages);
  for (uint32_t i = 0; i < S; ++i) mpk::mbar_init(bars + 8 * i, 1);
  mpk::mbar_init_fence();
  const uint64_t policy = s.hint ? mpk::l2_evict_first() : 0;

  const uint64_t first = blockIdx.x, step = gridDim.x;
  const uint64_t mine = first < ntiles ? (ntiles - 1 - first) / step + 1 : 0;  // this block's tiles
  auto issue_load = [&](uint64_t k) {
    const uint32_t st = static_cast<uint32_t>(k % S), bar = bars + 8 * st;
    const uint64_t tile = first + k * step;
    mpk::mbar_expect_tx(bar, s.stage_bytes + s.extra_tx);
    uint32_t off = base + st * s.stage_bytes;
    for (int i = 0; i < s.nload; ++i) {
      const uint8_t* src = s.load[i] + tile * s.load_bytes[i];
      if (s.hint)
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
            ::"r"(off), "l"(src), "r"(s.load_bytes[i]), "r"(bar), "l"(policy) : "memory");
      else
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(off), "l"(src), "r"(s.load_bytes[i]), "r"(bar) : "memory");
      off += s.load_bytes[i];
    }
  };

  uint64_t issued = 0, k = 0;
  for (; issued < mine && issued + 1 < S; ++issued) issue_load(issued);
  bool ok = true;
  for (; k < mine; ++k) {
    const uint32_t st = static_cast<uint32_t>(k % S);
    if (!mpk::mbar_wait(bars + 8 * st, static_cast<uint32_t>((k / S) & 1))) {
      ok = false;
      break;
    }
    const uint64_t tile = first + k * step;
    const uint32_t stage = base + st * s.stage_bytes;
    for (int j = 0; j < s.nstore; ++j) {
      uint8_t* dst = s.store[j] + tile * s.store_bytes[j];
      if (s.hint)
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
                     ::"l"(dst), "r"(stage + s.store_from[j]), "r"(s.store_bytes[j]), "l"(policy) : "memory");
      else
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                     ::"l"(dst), "r"(stage + s.store_from[j]), "r"(s.store_bytes[j]) : "memory");
    }
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    if (issued < mine) {
      // the stage of tile `issued` was last read by tile k - 1's stores:
      // wait until every store group but this tile's has read its data
      asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
      issue_load(issued++);
    }
  }
  if (!ok) {
    atomicExch(err, 1u);
    for (uint64_t j = k; j < issued; ++j)  // loads still in flight: bounded waits
      mpk::mbar_wait(bars + 8 * static_cast<uint32_t>(j % S), static_cast<uint32_t>((j / S) & 1));
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Launches bulk_streams_probe with blocks_per_sm blocks per SM; checks that
// they fit.
int launch_bulk(const BulkStreams& s, uint64_t ntiles, int blocks_per_sm, uint32_t* d_err, cudaStream_t stream) {
  if (s.stages < 2 || s.stages > kBulkMaxStages || blocks_per_sm < 1 || d_err == nullptr)
    return static_cast<int>(cudaErrorInvalidValue);
  const size_t smem = static_cast<size_t>(s.stages) * s.stage_bytes + 8u * static_cast<size_t>(s.stages);
  cudaError_t e = cudaFuncSetAttribute(bulk_streams_probe, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return static_cast<int>(e);
  int fit = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, bulk_streams_probe, 32, smem);
  if (e != cudaSuccess) return static_cast<int>(e);
  if (fit < blocks_per_sm) return static_cast<int>(cudaErrorInvalidConfiguration);
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return static_cast<int>(e);
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return static_cast<int>(e);
  bulk_streams_probe<<<sms * blocks_per_sm, 32, smem, stream>>>(s, ntiles, d_err);
  return static_cast<int>(cudaGetLastError());
}

bool aligned16(const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

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

// The step's streams over n parameters through TMA bulk copies, in tiles of
// `tile` parameters (a multiple of 64, so that a stage of tile * 14 bytes
// keeps the next one 128-B aligned; n a multiple of tile; every pointer 16-B
// aligned): blocks_per_sm blocks of one issuing thread per SM, `stages`
// stages each (2 .. 8, and they must fit in shared memory), hint 1 for an L2
// evict-first policy. *d_err (device) is set to 1 if a wait gave up. Returns
// a cudaError_t.
int mp_probe_step_streams_bulk_tile(uint16_t* params, const uint16_t* grads, float* master, float* m, float* v,
                                    uint64_t n, uint32_t tile, int blocks_per_sm, int stages, int hint,
                                    uint32_t* d_err, void* stream) {
  if (tile == 0 || tile % 64 || tile > (1u << 20) || n % tile || !aligned16(params) || !aligned16(grads) ||
      !aligned16(master) || !aligned16(m) || !aligned16(v))
    return static_cast<int>(cudaErrorInvalidValue);
  BulkStreams s{};
  s.nload = 4;
  s.load[0] = reinterpret_cast<const uint8_t*>(grads);
  s.load[1] = reinterpret_cast<const uint8_t*>(master);
  s.load[2] = reinterpret_cast<const uint8_t*>(m);
  s.load[3] = reinterpret_cast<const uint8_t*>(v);
  s.load_bytes[0] = tile * 2;
  s.load_bytes[1] = s.load_bytes[2] = s.load_bytes[3] = tile * 4;
  s.stage_bytes = tile * 14;
  s.nstore = 4;
  s.store[0] = reinterpret_cast<uint8_t*>(master);
  s.store[1] = reinterpret_cast<uint8_t*>(m);
  s.store[2] = reinterpret_cast<uint8_t*>(v);
  s.store[3] = reinterpret_cast<uint8_t*>(params);
  s.store_bytes[0] = s.store_bytes[1] = s.store_bytes[2] = tile * 4;
  s.store_bytes[3] = tile * 2;
  s.store_from[0] = tile * 2;   // master's staged tile
  s.store_from[1] = tile * 6;   // m's
  s.store_from[2] = tile * 10;  // v's
  s.store_from[3] = 0;          // the gradient's bits into the weight
  s.stages = stages;
  s.hint = hint ? 1 : 0;
  return launch_bulk(s, n / tile, blocks_per_sm, d_err, static_cast<cudaStream_t>(stream));
}

// mp_probe_step_streams_bulk_tile with 2048-parameter (28 KB) tiles.
int mp_probe_step_streams_bulk(uint16_t* params, const uint16_t* grads, float* master, float* m, float* v,
                               uint64_t n, int blocks_per_sm, int stages, int hint, uint32_t* d_err, void* stream) {
  return mp_probe_step_streams_bulk_tile(params, grads, master, m, v, n, kTile, blocks_per_sm, stages, hint, d_err,
                                         stream);
}

// dst <- src in `tiles` tiles of 28,672 B through TMA bulk copies (both
// pointers 16-B aligned; arguments otherwise as above).
int mp_probe_copy_bulk(void* dst, const void* src, uint64_t tiles, int blocks_per_sm, int stages, int hint,
                       uint32_t* d_err, void* stream) {
  if (!aligned16(dst) || !aligned16(src)) return static_cast<int>(cudaErrorInvalidValue);
  BulkStreams s{};
  s.nload = 1;
  s.load[0] = static_cast<const uint8_t*>(src);
  s.load_bytes[0] = s.stage_bytes = kTile * 14;
  s.nstore = 1;
  s.store[0] = static_cast<uint8_t*>(dst);
  s.store_bytes[0] = kTile * 14;
  s.store_from[0] = 0;
  s.stages = stages;
  s.hint = hint ? 1 : 0;
  return launch_bulk(s, tiles, blocks_per_sm, d_err, static_cast<cudaStream_t>(stream));
}

// The bulk copy probe over `tiles` 28,672-byte tiles of `buf` (dst = the
// second half) with every stage's mbarrier told to expect 16 bytes more than
// its loads bring: every load lands, but no stage's phase completes, so each
// block's bounded waits give up (one second each, for the wait and for the
// one load in flight) and set *d_err. For testing that give-up path; nothing
// faults or hangs. buf: device, 16-B aligned, 2 * tiles * 28,672 bytes.
int mp_probe_bulk_timeout(void* buf, uint64_t tiles, uint32_t* d_err, void* stream) {
  if (buf == nullptr || !aligned16(buf) || tiles == 0) return static_cast<int>(cudaErrorInvalidValue);
  BulkStreams s{};
  s.nload = 1;
  s.load[0] = static_cast<const uint8_t*>(buf);
  s.load_bytes[0] = s.stage_bytes = kTile * 14;
  s.nstore = 1;
  s.store[0] = static_cast<uint8_t*>(buf) + tiles * (kTile * 14);
  s.store_bytes[0] = kTile * 14;
  s.stages = 2;
  s.extra_tx = 16;
  return launch_bulk(s, tiles, 1, d_err, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
