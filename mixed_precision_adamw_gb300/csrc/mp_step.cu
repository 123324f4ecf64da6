// mp_step.cu — the fused AdamW + stochastic-rounding step kernels.
//
// llm.c walk-through ch. 04 "Multi-GPU and mixed precision" §2.2: one pass
// per parameter reads the bf16 gradient and the fp32 master/m/v, writes the
// fp32 master/m/v and the stochastically rounded bf16 weight. The step is
// bound by HBM traffic (28 B per parameter with master, 22 B without). Long
// ranges run adamw_tma_kernel, which stages whole tiles of every stream
// through shared memory with the TMA engine's bulk copies while its warps
// compute; other ranges run the register kernels, coalesced 16-B (fp32) and
// 8-B (bf16) vector streams in a grid-stride loop of persistent blocks sized
// to the SM count. All give the same bits. Weight decay comes from a
// per-launch table of decay segments (maximal runs of tensors with equal
// decay flag, §2.2's "2D tensors only").
#include <atomic>
#include <cmath>

#include "mp_device.cuh"
#include "mp_internal.h"
#include "mp_step.cuh"
#include "mp_tma.cuh"

namespace mpk {
namespace {

// Resident blocks per SM the register vector kernel is compiled for: the with-master
// kernel keeps 3 blocks of 256 threads (it compiles to 72 registers; forcing 4
// blocks, i.e. at most 64 registers, was 8 % slower on GB300); the no-master
// kernel moves fewer bytes per element and runs 9 % faster at 4 blocks (63
// registers), where the extra warps hide more memory latency.
template <bool kMaster>
struct VecOccupancy {
  static constexpr int kMinBlocks = kMaster ? 3 : 4;
};

// Vector path: the tiles of this block (vec_tiles in mp_step.cuh). kHead:
// the range starts mid-line and a head is peeled first (a separate
// instantiation, so that aligned ranges run the plain tile loop).
template <bool kMaster, uint32_t CAP, bool kDev, bool kHead>
__global__ void __launch_bounds__(kThreads, VecOccupancy<kMaster>::kMinBlocks)
adamw_vec_kernel(const __grid_constant__ StepArgs p, const __grid_constant__ SegTable<CAP> segs) {
  pdl_enter();
  float scale;
  if (!read_scale(p, scale)) return;
  uint32_t seed;
  const Hyper h = step_scalars<kDev>(p, seed);
  vec_tiles<kMaster, kHead>(p, segs, scale, h, seed, blockIdx.x, gridDim.x);
}

// Scalar path for buffers that are not vector-aligned: same arithmetic.
template <bool kMaster, uint32_t CAP, bool kDev>
__global__ void __launch_bounds__(kThreads)
adamw_scalar_kernel(const __grid_constant__ StepArgs p, const __grid_constant__ SegTable<CAP> segs) {
  pdl_enter();
  float scale;
  if (!read_scale(p, scale)) return;
  uint32_t seed;
  const Hyper h = step_scalars<kDev>(p, seed);
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
  uint64_t i = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x;
  Cursor c;
  c.s = seg_find(segs, p.nseg, p.goff + (i < p.n ? i : p.n - 1));
  c.end = segs.end[c.s];
  for (; i < p.n; i += stride) elem_update<kMaster>(p, segs, c, i, scale, h, seed);
}

// ---- TMA path ----------------------------------------------------------------
// One block per SM. Thread 0 (the producer) has the TMA engine load whole
// tiles of every input stream into a ring of shared-memory stages with 1D bulk
// copies and, once the consumer warps have updated a tile in place, store its
// results with bulk copies; the consumers run the register path's per-group
// update (stage_group). Tiles of a block: blockIdx.x + k*gridDim.x. Per stage
// two mbarriers: `full` (the tile's loads have landed: one arrival plus the
// expected bytes) and `done` (every consumer warp has written its share: one
// arrival per warp). A stage is loaded again only after the bulk stores of its
// previous tile have read it. Every wait gives up after one second and
// records MP_ERR_CUDA in *d_status; a block that gives up still waits,
// bounded, for its copies in flight before it ends.
//
// The shape was measured (interleaved builds, one launch of 201,326,592 params
// and the Llama-3-8B set's launches of 200,756,531): the streams reach their
// best rate in a narrow band of tile size, consumer warps and stages, e.g.
// with master 18 warps x 4 stages 6.78-6.81 TB/s, 17 x 4 6.65-6.68, 19 x 4
// 6.73-6.78, 18 x 3 5.77, 18 x 5 6.36-6.50; the register path 6.65-6.67.
// Larger tiles (two groups per consumer thread) did worse on the 8B update,
// 33.3 ms now: 18 x 3 of 4,608 params 33.6 ms, 16 x 3 of 4,096 34.4, and two
// stages of 4,608 or 6,144 params 52-61 ms, where the update of one tile no
// longer overlaps the loads of the next.
template <bool kMaster>
struct TmaConfig {
  static constexpr int kConsumerWarps = kMaster ? 18 : 26;
  static constexpr uint32_t kStages = kMaster ? 4 : 5;
  static constexpr int kConsumers = 32 * kConsumerWarps;
  static constexpr int kThreads = 32 + kConsumers;                        // one producer warp
  static constexpr uint32_t kTileElems = static_cast<uint32_t>(kConsumers) * kGroup;
  using Stage = TmaStage<kMaster, kTileElems>;
  static constexpr size_t kSmemBytes = kStages * Stage::kBytes + 16 * kStages;  // stages + 2 mbarriers each
};

__device__ __forceinline__ void tma_record_timeout(const StepArgs& p) {
  if (p.d_status != nullptr) atomicCAS(p.d_status, 0, MP_ERR_CUDA);
}

template <bool kMaster>
__device__ __noinline__ void tma_producer(const StepArgs& p, uint32_t base, uint32_t full, uint32_t done,
                                          uint64_t head, uint64_t mine) {
  using C = TmaConfig<kMaster>;
  using L = typename C::Stage;
  constexpr uint32_t S = C::kStages, T = C::kTileElems;
  const uint64_t pol = l2_evict_first();
  auto elem = [&](uint64_t k) { return head + (blockIdx.x + k * gridDim.x) * static_cast<uint64_t>(T); };
  auto load = [&](uint64_t k) {
    const uint32_t st = static_cast<uint32_t>(k % S), bar = full + 8 * st, sp = base + st * L::kBytes;
    const uint64_t e = elem(k);
    mbar_expect_tx(bar, L::kBytes);
    bulk_load(sp + L::kGrads, p.grads + e, T * 2, bar, pol);
    if constexpr (kMaster) bulk_load(sp + L::kW, p.master + e, T * 4, bar, pol);
    else bulk_load(sp + L::kW, p.params + e, T * 2, bar, pol);
    bulk_load(sp + L::kM, p.m + e, T * 4, bar, pol);
    bulk_load(sp + L::kV, p.v + e, T * 4, bar, pol);
  };
  uint64_t issued = 0, k = 0;
  for (; issued < mine && issued + 1 < S; ++issued) load(issued);
  bool ok = true;
  for (; k < mine; ++k) {
    const uint32_t st = static_cast<uint32_t>(k % S), sp = base + st * L::kBytes;
    if (!mbar_wait(done + 8 * st, static_cast<uint32_t>((k / S) & 1))) {
      ok = false;
      break;
    }
    const uint64_t e = elem(k);
    if constexpr (kMaster) {
      bulk_store(p.master + e, sp + L::kW, T * 4, pol);
      bulk_store(p.params + e, sp + L::kGrads, T * 2, pol);
    } else {
      bulk_store(p.params + e, sp + L::kW, T * 2, pol);
    }
    bulk_store(p.m + e, sp + L::kM, T * 4, pol);
    bulk_store(p.v + e, sp + L::kV, T * 4, pol);
    bulk_commit();
    if (issued < mine) {
      // the stage of tile `issued` last held tile k - 1: wait until every
      // store group but tile k's has read its data
      bulk_wait_read<1>();
      load(issued++);
    }
  }
  if (!ok) {
    tma_record_timeout(p);
    for (uint64_t j = k; j < issued; ++j)  // loads in flight: bounded waits
      mbar_wait(full + 8 * static_cast<uint32_t>(j % S), static_cast<uint32_t>((j / S) & 1));
  }
  bulk_wait_all();
}

template <bool kMaster, uint32_t CAP>
__global__ void __launch_bounds__(TmaConfig<kMaster>::kThreads, 1)
adamw_tma_kernel(const __grid_constant__ StepArgs p, const __grid_constant__ SegTable<CAP> segs) {
  pdl_enter();
  float scale;
  if (!read_scale(p, scale)) return;
  using C = TmaConfig<kMaster>;
  using L = typename C::Stage;
  constexpr uint32_t S = C::kStages, T = C::kTileElems;
  constexpr int kConsumers = C::kConsumers;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t base = smem_u32(smem);
  const uint32_t full = base + S * L::kBytes, done = full + 8 * S;
  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < S; ++i) {
      mbar_init(full + 8 * i, 1);
      mbar_init(done + 8 * i, C::kConsumerWarps);
    }
    mbar_init_fence();
  }
  __syncthreads();
  const uint64_t head = p.head < p.n ? p.head : p.n;
  const uint64_t ntiles = (p.n - head) / T;
  const uint64_t mine = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  if (threadIdx.x < 32) {
    if (threadIdx.x == 0) tma_producer<kMaster>(p, base, full, done, head, mine);
    return;
  }

  uint32_t seed;
  const Hyper h = step_scalars<false>(p, seed);
  const uint32_t ci = threadIdx.x - 32;
  const uint64_t lane0 = static_cast<uint64_t>(blockIdx.x) * kConsumers + ci;
  const uint64_t stride_tail = static_cast<uint64_t>(gridDim.x) * kConsumers;
  const uint64_t tail0 = head + ntiles * T + lane0;
  uint64_t first = mine ? head + static_cast<uint64_t>(blockIdx.x) * T + 4u * ci : tail0;
  if (lane0 < head) first = lane0;
  if (first >= p.n) first = p.n - 1;
  Cursor c;
  c.s = seg_find(segs, p.nseg, p.goff + first);
  c.end = segs.end[c.s];

  // head (the elements before the first tile), one element per thread
  for (uint64_t i = lane0; i < head; i += stride_tail) elem_update<kMaster>(p, segs, c, i, scale, h, seed);
  for (uint64_t k = 0; k < mine; ++k) {
    const uint32_t st = static_cast<uint32_t>(k % S);
    // every lane waits; the warp gives up as one, so its lanes stay together
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(full + 8 * st, static_cast<uint32_t>((k / S) & 1)))) {
      if ((threadIdx.x & 31) == 0) tma_record_timeout(p);
      break;
    }
    uint8_t* sp = smem + st * L::kBytes;
    const uint64_t e0 = head + (blockIdx.x + k * gridDim.x) * static_cast<uint64_t>(T);
#pragma unroll
    for (uint32_t g = ci; g < T / kGroup; g += kConsumers)
      stage_group<kMaster, T>(p, segs, c, sp, g, e0, scale, h, seed);
    fence_to_bulk();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(done + 8 * st);
  }
  // ragged tail (< T elements), one element per thread
  for (uint64_t i = tail0; i < p.n; i += stride_tail) elem_update<kMaster>(p, segs, c, i, scale, h, seed);
}

// Resident blocks per SM of `kernel` on `device`, queried once. `cache` must
// belong to that one kernel: the with- and no-master instantiations share a
// function-pointer type but not their register counts.
template <typename K>
int blocks_per_sm(K kernel, int device, std::atomic<int> (&cache)[64]) {
  const bool cached = device >= 0 && device < 64;
  int nb = cached ? cache[device].load(std::memory_order_relaxed) : 0;  // 0 = not yet queried
  if (nb == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, kThreads, 0) != cudaSuccess || nb < 1) {
      cudaGetLastError();  // clear the query's error; the launch reports its own
      return 1;            // not cached: the next call asks again
    }
    if (cached) cache[device].store(nb, std::memory_order_relaxed);  // racing callers store the same value
  }
  return nb;
}

template <bool kMaster, uint32_t CAP, bool kDev>
cudaError_t launch_cap(const StepArgs& a, const uint64_t* seg_end, bool vec, const DeviceInfo& dev,
                       cudaStream_t stream) {
  SegTable<CAP> t;
  for (uint32_t s = 0; s < a.nseg; ++s) t.end[s] = seg_end[s];
  for (uint32_t s = a.nseg; s < CAP; ++s) t.end[s] = seg_end[a.nseg - 1];
  // one cache per kernel: <kMaster, CAP, kDev> and the vector kernel's kHead
  static std::atomic<int> vec_occupancy[64], vec_head_occupancy[64], scalar_occupancy[64];
  if (vec && !kDev) {
    // The TMA path, for ranges of at least two tiles per SM whose tiles start
    // 16-B aligned in every array (bulk copies need it), after the head that
    // brings the gradients to their next 128-B line.
    const uint32_t head = static_cast<uint32_t>(((128u - (reinterpret_cast<uintptr_t>(a.grads) & 127u)) & 127u) / 2u);
    using C = TmaConfig<kMaster>;
    const uint64_t grid = static_cast<uint64_t>(dev.sms);
    const bool fits = static_cast<uint64_t>(head) < a.n && (a.n - head) / C::kTileElems >= 2 * grid;
    const bool aligned = reinterpret_cast<uintptr_t>(a.params + head) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(a.m + head) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(a.v + head) % 16 == 0 &&
                         (!kMaster || reinterpret_cast<uintptr_t>(a.master + head) % 16 == 0);
    if (fits && aligned) {
      static std::atomic<bool> smem_set[64];
      auto k = adamw_tma_kernel<kMaster, CAP>;
      constexpr size_t smem = C::kSmemBytes;
      const bool cached = dev.device >= 0 && dev.device < 64;
      if (!cached || !smem_set[dev.device].load(std::memory_order_relaxed)) {
        const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        if (cached) smem_set[dev.device].store(true, std::memory_order_relaxed);
      }
      StepArgs b = a;
      b.head = head;
      const uint64_t ntiles = (a.n - head) / C::kTileElems;
      const uint64_t blocks = ntiles < grid ? ntiles : grid;
      return launch_pdl_smem(k, static_cast<unsigned>(blocks), C::kThreads, smem, stream, b, t);
    }
  }
  if (vec) {
    // Peel the elements before the gradients' next 128-B line (a multiple of
    // 4 below 64, as grads are 8-B aligned), so that the tiles' vectors start
    // on whole lines: a range that starts mid-line (a shard of a size that
    // is not a multiple of 64) would otherwise split every warp's accesses
    // across an extra line.
    StepArgs b = a;
    const uint32_t head = static_cast<uint32_t>(((128u - (reinterpret_cast<uintptr_t>(a.grads) & 127u)) & 127u) / 2u);
    b.head = static_cast<uint64_t>(head) < a.n ? head : static_cast<uint32_t>(a.n);
    const uint64_t ntiles = (b.n - b.head) / kTile;
    auto k = b.head ? adamw_vec_kernel<kMaster, CAP, kDev, true> : adamw_vec_kernel<kMaster, CAP, kDev, false>;
    const uint64_t cap = static_cast<uint64_t>(dev.sms) *
                         blocks_per_sm(k, dev.device, b.head ? vec_head_occupancy : vec_occupancy);
    uint64_t blocks = ntiles ? ntiles : (b.n + kThreads - 1) / kThreads;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(k, static_cast<unsigned>(blocks), kThreads, stream, b, t);
  } else {
    auto k = adamw_scalar_kernel<kMaster, CAP, kDev>;
    const uint64_t cap = static_cast<uint64_t>(dev.sms) * blocks_per_sm(k, dev.device, scalar_occupancy);
    uint64_t blocks = (a.n + kThreads - 1) / kThreads;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(k, static_cast<unsigned>(blocks), kThreads, stream, a, t);
  }
}

}  // namespace

cudaError_t launch_adamw(const StepArgs& a, const uint64_t* seg_end, bool vec, const DeviceInfo& dev,
                         cudaStream_t stream) {
  const bool master = a.master != nullptr;
  if (a.dstate != nullptr)  // replayable steps: one segment capacity is enough
    return master ? launch_cap<true, kSegCapLarge, true>(a, seg_end, vec, dev, stream)
                  : launch_cap<false, kSegCapLarge, true>(a, seg_end, vec, dev, stream);
  if (a.nseg <= kSegCapSmall)
    return master ? launch_cap<true, kSegCapSmall, false>(a, seg_end, vec, dev, stream)
                  : launch_cap<false, kSegCapSmall, false>(a, seg_end, vec, dev, stream);
  return master ? launch_cap<true, kSegCapLarge, false>(a, seg_end, vec, dev, stream)
                : launch_cap<false, kSegCapLarge, false>(a, seg_end, vec, dev, stream);
}

}  // namespace mpk
