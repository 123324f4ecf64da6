// mp_small.cu — the whole optimizer step in one launch for small parameter
// sets.
//
// llm.c walk-through ch. 04 "Multi-GPU and mixed precision" §4 gives the
// train-step order (global grad norm, clip scale, outlier check, update) and
// §2.2 the update. For a buffer of a few tens of thousands of parameters the
// general path's three launches (norm partials, norm finalize, update) cost
// more than the work. Here one thread-block cluster of 16 CTAs does it all:
// every CTA first issues the loads of its update inputs (they do not depend
// on the norm) and computes one norm partial; at a hardware cluster barrier
// the partials become visible to the whole cluster, and every CTA reads them
// out of the other CTAs' shared memory (distributed shared memory) and adds
// them with the finalize kernel's bits (small_total), so all CTAs hold the
// same norm and clip scale and finish their updates with no further
// barrier; CTA 0 writes the norm, the scale and the step count. With the outlier check, which
// updates its window in one thread, CTA 0 alone derives the norm, runs the
// check and hands the scale to the cluster through a second barrier. The
// results are the general path's bit for bit: CTA r computes the partial of
// norm block r of the general path's norm grid with the same code
// (mp_norm.cuh), the partials are added to the finalize kernel's bits, and
// the update is the general path's tile and element code (mp_step.cuh). All
// waits are cluster barriers; the launch co-schedules the cluster's CTAs.
#include <cooperative_groups.h>

#include <atomic>
#include <cmath>

#include "mp_adamw.h"
#include "mp_device.cuh"
#include "mp_internal.h"
#include "mp_norm.cuh"
#include "mp_outlier.cuh"
#include "mp_step.cuh"

namespace cg = cooperative_groups;

namespace mpk {
namespace {

// What CTA 0 hands to the cluster after the outlier check: the clip scale
// and the step's learning rate, bias corrections and rounding seed.
struct StepScalars {
  float scale, lr, bc1, bc2;
  uint32_t seed;
};

// The finalize kernel's total of nb <= 32 partials, from warp 0 alone. In
// the finalize kernel (norm_total) thread i < nb holds partial i and every
// other thread 0.0; the first level of the block sum is the shuffle tree of
// each warp, so warp 0 forms exactly the tree computed here, the other warps
// form +0.0, and the second level adds only those zeros to warp 0's sum,
// which changes nothing (x + 0 = x for every partial sum x >= +0, NaN and
// Inf included). The same bits, with no second level and one barrier.
template <typename PartialAt>
__device__ __forceinline__ double small_total(PartialAt partial, int nb, double* sh) {
  if (threadIdx.x < 32) {
    double d = static_cast<int>(threadIdx.x) < nb ? __dadd_rn(0.0, partial(threadIdx.x)) : 0.0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) d = __dadd_rn(d, __shfl_down_sync(0xFFFFFFFFu, d, o));
    if (threadIdx.x == 0) sh[0] = d;
  }
  __syncthreads();
  return sh[0];
}

// CTA r updates tile r (if r < n / kTile) and, one element per thread, the
// tail element n / kTile * kTile + r * kThreads + t (if below n): the
// general path's mapping for a grid of kSmallClusterCtas blocks when there
// is at most one tile per block.
template <bool kMaster>
__global__ void __launch_bounds__(kThreads)
small_step_kernel(const __grid_constant__ StepArgs p, const __grid_constant__ SmallArgs a,
                  const __grid_constant__ SegTable<kSegCapSmall> segs) {
  __shared__ double sh[kThreads / 32 + 1];
  __shared__ double partial;
  __shared__ StepScalars out;
  pdl_enter();
  const cg::cluster_group cluster = cg::this_cluster();
  const uint32_t rank = cluster.block_rank();
  const bool lead = rank == 0 && threadIdx.x == 0;

  // 0. The update's inputs, loaded now so that their latency overlaps the
  // norm. Gradients are read where the norm reads them (host memory in the
  // copy case: the same values as the device copy the norm writes). The
  // step counter is read before the first barrier, after which CTA 0 may
  // advance it.
  const uint64_t ntiles = p.n / kTile;
  const bool has_tile = rank < ntiles;
  const uint64_t e0 = static_cast<uint64_t>(rank) * kTile + threadIdx.x * kGroup;
  const uint64_t ti = ntiles * kTile + static_cast<uint64_t>(rank) * kThreads + threadIdx.x;
  const bool has_tail = ti < p.n;
  TileIn tin;
  ElemIn ein;
  if (has_tile) load_tile<kMaster>(p, a.norm_src, e0, tin);
  if (has_tail) load_elem<kMaster>(p, a.norm_src, ti, ein);
  ClockStep cs{0, p.seed, p.bc1, p.bc2, p.lr, true};
  if (a.clock.state != nullptr) cs = next_clock_step(a.clock);
  Cursor c;  // decay segment of this thread's first element
  c.s = seg_find(segs, p.nseg, p.goff + (has_tile ? e0 : (has_tail ? ti : p.n - 1)));
  c.end = segs.end[c.s];

  // 1. Norm block `rank` of the general path's grid.
  if (rank < static_cast<uint32_t>(a.nb)) {
    const double S = a.copy_out != nullptr
                         ? norm_block_partial<true>(a.norm_src, p.n, a.norm_vec, a.copy_out, rank, a.nb, sh)
                         : norm_block_partial<false>(a.norm_src, p.n, a.norm_vec, nullptr, rank, a.nb, sh);
    if (threadIdx.x == 0) partial = S;
  }
  cluster.sync();

  float scale;
  if (a.outlier == nullptr) {
    // 2a. Every CTA adds the partials in the finalize kernel's order (the
    // same total everywhere); CTA 0 records the step. Other CTAs' shared
    // memory is read only here: arrive now, wait before exiting. The arrive
    // needs no release: every value read has been used by the sum.
    const double S = small_total([&](int i) { return *cluster.map_shared_rank(&partial, i); }, a.nb, sh);
    __cluster_barrier_arrive_relaxed();
    // One thread takes the fp64 square root (fp64 is a small fraction of the
    // fp32 rate on this GPU) and shares the scale through shared memory.
    if (threadIdx.x == 0) {
      float norm, sc;
      norm_and_scale(S, a.clip, norm, sc);
      if (!cs.ok) sc = __int_as_float(0x7FC00000);
      if (lead) {
        if (a.clock.state != nullptr) {
          if (cs.ok) commit_clock_step(a.clock, cs);
          else if (a.clock.d_status != nullptr) atomicCAS(a.clock.d_status, 0, MP_ERR_RANGE);
        }
        *a.d_norm = norm;
        *a.d_scale = sc;
        if (!isfinite(sc) && p.d_status != nullptr) atomicCAS(p.d_status, 0, MP_ERR_NONFINITE);
      }
      out.scale = sc;
    }
    __syncthreads();
    scale = out.scale;
    if (isfinite(scale)) {
      const Hyper h{cs.lr, p.beta1, p.beta2, p.eps, p.wd, cs.bc1, cs.bc2};
      if (has_tile) update_tile<kMaster>(p, segs, c, e0, tin, scale, h, cs.seed);
      if (has_tail) update_elem<kMaster>(p, segs, c, ti, ein, scale, h, cs.seed);
    }
    __cluster_barrier_wait();
    return;
  }

  // 2b. With the outlier check (one thread, it updates the window): CTA 0
  // derives the norm, records the step, runs the check in the general path's
  // order and hands the scalars to the cluster.
  if (rank == 0) {
    const double S = small_total([&](int i) { return *cluster.map_shared_rank(&partial, i); }, a.nb, sh);
    if (threadIdx.x == 0) {
      float norm;
      norm_and_scale(S, a.clip, norm, scale);
      if (a.clock.state != nullptr) {
        if (cs.ok) commit_clock_step(a.clock, cs);
        else {
          scale = __int_as_float(0x7FC00000);
          if (a.clock.d_status != nullptr) atomicCAS(a.clock.d_status, 0, MP_ERR_RANGE);
        }
      }
      *a.d_norm = norm;
      if (outlier_update(static_cast<OutlierState*>(a.outlier), norm, a.outlier_z, a.d_z, p.d_status))
        scale = __int_as_float(0x7FC00000);
      *a.d_scale = scale;
      if (!isfinite(scale) && p.d_status != nullptr) atomicCAS(p.d_status, 0, MP_ERR_NONFINITE);
      out = StepScalars{scale, cs.lr, cs.bc1, cs.bc2, cs.seed};
    }
  }
  cluster.sync();

  // 3. Every CTA: the scalars from CTA 0, then its update. CTA 0's shared
  // memory must stay alive until every CTA has read it: arrive now, wait
  // before exiting.
  const StepScalars o = *cluster.map_shared_rank(&out, 0);
  auto token = cluster.barrier_arrive();
  if (isfinite(o.scale)) {
    const Hyper h{o.lr, p.beta1, p.beta2, p.eps, p.wd, o.bc1, o.bc2};
    if (has_tile) update_tile<kMaster>(p, segs, c, e0, tin, o.scale, h, o.seed);
    if (has_tail) update_elem<kMaster>(p, segs, c, ti, ein, o.scale, h, o.seed);
  }
  cluster.barrier_wait(std::move(token));
}

cudaLaunchConfig_t small_config(cudaLaunchAttribute (&attr)[2], cudaStream_t stream) {
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kSmallClusterCtas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kSmallClusterCtas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

// 16 CTAs exceed the portable cluster size of 8: the kernel must opt in, and
// the GPU must be able to place such a cluster. 0 = not yet asked, 1 = yes,
// -1 = no; racing first calls store the same answer.
template <bool kMaster>
bool available(int device) {
  static std::atomic<int> answer[64];
  if (device < 0 || device >= 64) return false;
  int known = answer[device].load(std::memory_order_relaxed);
  if (known == 0) {
    int size = 0;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = small_config(attr, nullptr);
    cfg.numAttrs = 0;  // the query takes the cluster size from the kernel's limits
    bool ok = cudaFuncSetAttribute(small_step_kernel<kMaster>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                   1) == cudaSuccess &&
              cudaOccupancyMaxPotentialClusterSize(&size, small_step_kernel<kMaster>, &cfg) == cudaSuccess &&
              size >= kSmallClusterCtas;
    if (!ok) cudaGetLastError();  // clear a non-sticky error of the queries
    known = ok ? 1 : -1;
    answer[device].store(known, std::memory_order_relaxed);
  }
  return known > 0;
}

}  // namespace

bool small_step_available(const DeviceInfo& dev, bool master) {
  return master ? available<true>(dev.device) : available<false>(dev.device);
}

cudaError_t launch_small_step(const StepArgs& a, const SmallArgs& s, const uint64_t* seg_end,
                              cudaStream_t stream) {
  SegTable<kSegCapSmall> t;
  for (uint32_t i = 0; i < a.nseg; ++i) t.end[i] = seg_end[i];
  for (uint32_t i = a.nseg; i < kSegCapSmall; ++i) t.end[i] = seg_end[a.nseg - 1];
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = small_config(attr, stream);
  return a.master != nullptr ? cudaLaunchKernelEx(&cfg, small_step_kernel<true>, a, s, t)
                             : cudaLaunchKernelEx(&cfg, small_step_kernel<false>, a, s, t);
}

}  // namespace mpk
