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
#include <cmath>

#include "mp_device.cuh"
#include "mp_internal.h"

namespace mpk {
namespace {

template <uint32_t CAP>
struct SegTable {
  unsigned long long end[CAP];
};

struct Cursor {
  uint32_t s;
  unsigned long long end;
};

template <uint32_t CAP>
__device__ __forceinline__ uint32_t seg_find(const SegTable<CAP>& t, uint32_t nseg, uint64_t gi) {
  uint32_t lo = 0, hi = nseg - 1;  // smallest s with end[s] > gi (end[nseg-1] > gi)
  while (lo < hi) {
    const uint32_t mid = (lo + hi) >> 1;
    if (t.end[mid] > gi) hi = mid; else lo = mid + 1;
  }
  return lo;
}

// Moves the cursor forward to the segment holding gi. gi only grows along a
// thread's iterations and is always < end[nseg-1], so this never runs past
// the table.
template <uint32_t CAP>
__device__ __forceinline__ void seek(Cursor& c, const SegTable<CAP>& t, uint64_t gi) {
  while (gi >= c.end) {
    ++c.s;
    c.end = t.end[c.s];
  }
}

__device__ __forceinline__ float seg_wd(const StepArgs& p, uint32_t s) {
  return ((p.first_decay ^ s) & 1u) ? p.wd : 0.0f;
}

template <uint32_t CAP>
__device__ __forceinline__ void group_decay(Cursor& c, const SegTable<CAP>& t, const StepArgs& p,
                                            uint64_t gi, float (&wd)[kGroup]) {
  seek(c, t, gi);
  if (gi + kGroup <= c.end) {
    const float w = seg_wd(p, c.s);
#pragma unroll
    for (int j = 0; j < kGroup; ++j) wd[j] = w;
  } else {  // the group straddles a segment boundary
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      seek(c, t, gi + j);
      wd[j] = seg_wd(p, c.s);
    }
  }
}

// The launch's hyperparameters and rounding seed; with kDev, the per-step
// ones (lr, bias corrections, seed) come from the device step state.
template <bool kDev>
__device__ __forceinline__ Hyper step_scalars(const StepArgs& p, uint32_t& seed) {
  Hyper h{p.lr, p.beta1, p.beta2, p.eps, p.wd, p.bc1, p.bc2};
  seed = p.seed;
  if (kDev) {
    const mp_step_state_t* s = p.dstate;
    h.lr = s->lr;
    h.bc1 = s->bc1;
    h.bc2 = s->bc2;
    seed = s->seed;
  }
  return h;
}

// Updates 4 consecutive elements starting at global index gi.
__device__ __forceinline__ uint2 group_update(uint2 graw, float4& m4, float4& v4, float (&w)[kGroup],
                                              const float (&wd)[kGroup], float scale, const Hyper& h,
                                              uint64_t gi, uint32_t seed) {
  const float g[kGroup] = {bf16_lo(graw.x), bf16_hi(graw.x), bf16_lo(graw.y), bf16_hi(graw.y)};
  float mm[kGroup] = {m4.x, m4.y, m4.z, m4.w};
  float vv[kGroup] = {v4.x, v4.y, v4.z, v4.w};
  uint32_t r[kGroup], pos[kGroup];
  noise_pos4(gi, pos);
#pragma unroll
  for (int j = 0; j < kGroup; ++j) {
    w[j] = adamw_update(g[j], mm[j], vv[j], w[j], wd[j], scale, h);
    r[j] = sr_bf16_c(w[j], draw16_complement(pos[j], seed));
  }
  m4 = make_float4(mm[0], mm[1], mm[2], mm[3]);
  v4 = make_float4(vv[0], vv[1], vv[2], vv[3]);
  return make_uint2(r[0] | (r[1] << 16), r[2] | (r[3] << 16));
}

template <bool kMaster, uint32_t CAP>
__device__ __forceinline__ void elem_update(const StepArgs& p, const SegTable<CAP>& t, Cursor& c,
                                            uint64_t i, float scale, const Hyper& h, uint32_t seed) {
  const uint64_t gi = p.goff + i;
  seek(c, t, gi);
  float m = p.m[i];
  float v = p.v[i];
  const float old = kMaster ? p.master[i] : bf16_to_f32(p.params[i]);
  const float w = adamw_update(bf16_to_f32(p.grads[i]), m, v, old, seg_wd(p, c.s), scale, h);
  p.m[i] = m;
  p.v[i] = v;
  if (kMaster) p.master[i] = w;
  p.params[i] = static_cast<uint16_t>(sr_bf16_c(w, draw16_complement(noise_pos(gi), seed)));
}

// Reads the clip scale; a non-finite scale stops every thread before any
// write (the decision is uniform: all threads read the same value).
__device__ __forceinline__ bool read_scale(const StepArgs& p, float& scale) {
  scale = (p.d_scale != nullptr) ? *p.d_scale : 1.0f;
  if (!isfinite(scale)) {
    // MP_ERR_NONFINITE, unless an earlier error (e.g. an outlier skip) is already recorded
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.d_status != nullptr) atomicCAS(p.d_status, 0, 5);
    return false;
  }
  return true;
}

// Resident blocks per SM the vector kernel is compiled for: the with-master
// kernel keeps 3 blocks of 256 threads (it compiles to 72 registers; forcing 4
// blocks, i.e. at most 64 registers, was 8 % slower on GB300); the no-master
// kernel moves fewer bytes per element and runs 9 % faster at 4 blocks (63
// registers), where the extra warps hide more memory latency.
template <bool kMaster>
struct VecOccupancy {
  static constexpr int kMinBlocks = kMaster ? 3 : 4;
};

// Vector path: requires params/grads 8-B aligned and master/m/v 16-B aligned.
// Block-iteration k covers tile k of kTile elements; thread t handles the two
// 4-element groups at tile offsets 4t and 4t + 4*kThreads, so every warp-wide
// load or store is one contiguous 512-B (fp32) or 256-B (bf16) span.
template <bool kMaster, uint32_t CAP, bool kDev>
__global__ void __launch_bounds__(kThreads, VecOccupancy<kMaster>::kMinBlocks)
adamw_vec_kernel(const __grid_constant__ StepArgs p, const __grid_constant__ SegTable<CAP> segs) {
  pdl_enter();
  float scale;
  if (!read_scale(p, scale)) return;
  uint32_t seed;
  const Hyper h = step_scalars<kDev>(p, seed);
  const uint64_t ntiles = p.n / kTile;
  const uint64_t stride_tail = static_cast<uint64_t>(gridDim.x) * kThreads;
  const uint64_t tail0 = ntiles * kTile + static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x;
  uint64_t first = (blockIdx.x < ntiles) ? static_cast<uint64_t>(blockIdx.x) * kTile + threadIdx.x * kGroup
                                         : tail0;
  if (first >= p.n) first = p.n - 1;
  Cursor c;
  c.s = seg_find(segs, p.nseg, p.goff + first);
  c.end = segs.end[c.s];

  for (uint64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const uint64_t e0 = tile * kTile + threadIdx.x * kGroup;
    const uint64_t e1 = e0 + kThreads * kGroup;
    const uint2 g0 = __ldcs(reinterpret_cast<const uint2*>(p.grads + e0));
    const uint2 g1 = __ldcs(reinterpret_cast<const uint2*>(p.grads + e1));
    float4 m0 = __ldcs(reinterpret_cast<const float4*>(p.m + e0));
    float4 m1 = __ldcs(reinterpret_cast<const float4*>(p.m + e1));
    float4 v0 = __ldcs(reinterpret_cast<const float4*>(p.v + e0));
    float4 v1 = __ldcs(reinterpret_cast<const float4*>(p.v + e1));
    float w0[kGroup], w1[kGroup];
    if (kMaster) {
      const float4 a = __ldcs(reinterpret_cast<const float4*>(p.master + e0));
      const float4 b = __ldcs(reinterpret_cast<const float4*>(p.master + e1));
      w0[0] = a.x; w0[1] = a.y; w0[2] = a.z; w0[3] = a.w;
      w1[0] = b.x; w1[1] = b.y; w1[2] = b.z; w1[3] = b.w;
    } else {
      const uint2 a = __ldcs(reinterpret_cast<const uint2*>(p.params + e0));
      const uint2 b = __ldcs(reinterpret_cast<const uint2*>(p.params + e1));
      w0[0] = bf16_lo(a.x); w0[1] = bf16_hi(a.x); w0[2] = bf16_lo(a.y); w0[3] = bf16_hi(a.y);
      w1[0] = bf16_lo(b.x); w1[1] = bf16_hi(b.x); w1[2] = bf16_lo(b.y); w1[3] = bf16_hi(b.y);
    }
    float wd0[kGroup], wd1[kGroup];
    group_decay(c, segs, p, p.goff + e0, wd0);
    group_decay(c, segs, p, p.goff + e1, wd1);

    const uint2 q0 = group_update(g0, m0, v0, w0, wd0, scale, h, p.goff + e0, seed);
    const uint2 q1 = group_update(g1, m1, v1, w1, wd1, scale, h, p.goff + e1, seed);

    __stcs(reinterpret_cast<float4*>(p.m + e0), m0);
    __stcs(reinterpret_cast<float4*>(p.m + e1), m1);
    __stcs(reinterpret_cast<float4*>(p.v + e0), v0);
    __stcs(reinterpret_cast<float4*>(p.v + e1), v1);
    if (kMaster) {
      __stcs(reinterpret_cast<float4*>(p.master + e0), make_float4(w0[0], w0[1], w0[2], w0[3]));
      __stcs(reinterpret_cast<float4*>(p.master + e1), make_float4(w1[0], w1[1], w1[2], w1[3]));
    }
    __stcs(reinterpret_cast<uint2*>(p.params + e0), q0);
    __stcs(reinterpret_cast<uint2*>(p.params + e1), q1);
  }
  // Ragged tail (< kTile elements), one element per thread.
  for (uint64_t i = tail0; i < p.n; i += stride_tail) elem_update<kMaster>(p, segs, c, i, scale, h, seed);
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
int blocks_per_sm(K kernel, int device, int (&cache)[64]) {
  if (device < 0 || device >= 64) device = 0;
  int nb = cache[device];  // 0 = not yet queried; racing writers store the same value
  if (nb == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel, kThreads, 0) != cudaSuccess || nb < 1) nb = 1;
    cache[device] = nb;
  }
  return nb;
}

template <bool kMaster, uint32_t CAP, bool kDev>
cudaError_t launch_cap(const StepArgs& a, const uint64_t* seg_end, bool vec, const DeviceInfo& dev,
                       cudaStream_t stream) {
  SegTable<CAP> t;
  for (uint32_t s = 0; s < a.nseg; ++s) t.end[s] = seg_end[s];
  for (uint32_t s = a.nseg; s < CAP; ++s) t.end[s] = seg_end[a.nseg - 1];
  static int vec_occupancy[64], scalar_occupancy[64];  // one cache per <kMaster, CAP, kDev> kernel
  const uint64_t ntiles = a.n / kTile;
  if (vec) {
    auto k = adamw_vec_kernel<kMaster, CAP, kDev>;
    const uint64_t cap = static_cast<uint64_t>(dev.sms) * blocks_per_sm(k, dev.device, vec_occupancy);
    uint64_t blocks = ntiles ? ntiles : (a.n + kThreads - 1) / kThreads;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    return launch_pdl(k, static_cast<unsigned>(blocks), kThreads, stream, a, t);
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
