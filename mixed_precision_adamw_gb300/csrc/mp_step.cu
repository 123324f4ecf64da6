// mp_step.cu — the fused AdamW + stochastic-rounding step kernel.
//
// llm.c walk-through ch. 04 "Multi-GPU and mixed precision" §2.2: one pass
// per parameter reads the bf16 gradient and the fp32 master/m/v, writes the
// fp32 master/m/v and the stochastically rounded bf16 weight. The kernel is
// bound by HBM traffic (28 B per parameter with master, 22 B without), so it
// is written as coalesced 16-B (fp32) and 8-B (bf16) vector streams over all
// arrays in one pass, in a grid-stride loop of persistent blocks sized to the
// SM count. Weight decay comes from a per-launch table of decay segments
// (maximal runs of tensors with equal decay flag, §2.2's "2D tensors only").
#include <atomic>
#include <cmath>

#include "mp_device.cuh"
#include "mp_internal.h"
#include "mp_step.cuh"

namespace mpk {
namespace {

// Resident blocks per SM the vector kernel is compiled for: the with-master
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
