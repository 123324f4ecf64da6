// mp_step.cuh — device building blocks of the AdamW + stochastic-rounding
// step, shared by the step kernels (mp_step.cu) and the one-launch step for
// small parameter sets (mp_small.cu).
//
// llm.c walk-through ch. 04 "Multi-GPU and mixed precision" §2.2: one pass
// per parameter reads the bf16 gradient and the fp32 master/m/v, writes the
// fp32 master/m/v and the stochastically rounded bf16 weight; weight decay
// applies to 2D tensors only, here through a table of decay segments
// (maximal runs of tensors with equal decay flag).
#pragma once

#include <cstdint>

#include "mp_device.cuh"
#include "mp_internal.h"

namespace mpk {

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
    r[j] = sr_bf16_hi(w[j], draw16_complement(pos[j], seed));
  }
  m4 = make_float4(mm[0], mm[1], mm[2], mm[3]);
  v4 = make_float4(vv[0], vv[1], vv[2], vv[3]);
  return make_uint2(pack_hi16(r[0], r[1]), pack_hi16(r[2], r[3]));
}

// Updates 4 consecutive elements: m, v and the new fp32 weights w (the
// rounding is left to the caller).
__device__ __forceinline__ void group_update_only(uint2 graw, float4& m4, float4& v4, float (&w)[kGroup],
                                                  const float (&wd)[kGroup], float scale, const Hyper& h) {
  const float g[kGroup] = {bf16_lo(graw.x), bf16_hi(graw.x), bf16_lo(graw.y), bf16_hi(graw.y)};
  float mm[kGroup] = {m4.x, m4.y, m4.z, m4.w};
  float vv[kGroup] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
  for (int j = 0; j < kGroup; ++j) w[j] = adamw_update(g[j], mm[j], vv[j], w[j], wd[j], scale, h);
  m4 = make_float4(mm[0], mm[1], mm[2], mm[3]);
  v4 = make_float4(vv[0], vv[1], vv[2], vv[3]);
}

// One element's inputs: its gradient, m, v and old weight.
struct ElemIn {
  float g, m, v, old;
};

// Loads element i's inputs; the gradient from `grads` (p.grads, or another
// copy of the same values).
template <bool kMaster>
__device__ __forceinline__ void load_elem(const StepArgs& p, const uint16_t* grads, uint64_t i, ElemIn& in) {
  in.m = p.m[i];
  in.v = p.v[i];
  in.old = kMaster ? p.master[i] : bf16_to_f32(p.params[i]);
  in.g = bf16_to_f32(grads[i]);
}

// Updates element i from its loaded inputs and stores the results.
template <bool kMaster, uint32_t CAP>
__device__ __forceinline__ void update_elem(const StepArgs& p, const SegTable<CAP>& t, Cursor& c, uint64_t i,
                                            ElemIn& in, float scale, const Hyper& h, uint32_t seed) {
  const uint64_t gi = p.goff + i;
  seek(c, t, gi);
  const float w = adamw_update(in.g, in.m, in.v, in.old, seg_wd(p, c.s), scale, h);
  p.m[i] = in.m;
  p.v[i] = in.v;
  if (kMaster) p.master[i] = w;
  p.params[i] = static_cast<uint16_t>(sr_bf16_c(w, draw16_complement(noise_pos(gi), seed)));
}

template <bool kMaster, uint32_t CAP>
__device__ __forceinline__ void elem_update(const StepArgs& p, const SegTable<CAP>& t, Cursor& c,
                                            uint64_t i, float scale, const Hyper& h, uint32_t seed) {
  ElemIn in;
  load_elem<kMaster>(p, p.grads, i, in);
  update_elem<kMaster>(p, t, c, i, in, scale, h, seed);
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

// One thread's share of a tile: the two 4-element groups at tile offsets 4t
// and 4t + 4*kThreads (e0 and e0 + 4*kThreads below).
struct TileIn {
  uint2 g0, g1;
  float4 m0, m1, v0, v1;
  float w0[kGroup], w1[kGroup];
};

// Issues the 8 vector loads of a thread's share of the tile at e0; the
// gradients from `grads` (p.grads, or another copy of the same values).
template <bool kMaster>
__device__ __forceinline__ void load_tile(const StepArgs& p, const uint16_t* grads, uint64_t e0, TileIn& in) {
  const uint64_t e1 = e0 + kThreads * kGroup;
  in.g0 = __ldcs(reinterpret_cast<const uint2*>(grads + e0));
  in.g1 = __ldcs(reinterpret_cast<const uint2*>(grads + e1));
  in.m0 = __ldcs(reinterpret_cast<const float4*>(p.m + e0));
  in.m1 = __ldcs(reinterpret_cast<const float4*>(p.m + e1));
  in.v0 = __ldcs(reinterpret_cast<const float4*>(p.v + e0));
  in.v1 = __ldcs(reinterpret_cast<const float4*>(p.v + e1));
  if (kMaster) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(p.master + e0));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(p.master + e1));
    in.w0[0] = a.x; in.w0[1] = a.y; in.w0[2] = a.z; in.w0[3] = a.w;
    in.w1[0] = b.x; in.w1[1] = b.y; in.w1[2] = b.z; in.w1[3] = b.w;
  } else {
    const uint2 a = __ldcs(reinterpret_cast<const uint2*>(p.params + e0));
    const uint2 b = __ldcs(reinterpret_cast<const uint2*>(p.params + e1));
    in.w0[0] = bf16_lo(a.x); in.w0[1] = bf16_hi(a.x); in.w0[2] = bf16_lo(a.y); in.w0[3] = bf16_hi(a.y);
    in.w1[0] = bf16_lo(b.x); in.w1[1] = bf16_hi(b.x); in.w1[2] = bf16_lo(b.y); in.w1[3] = bf16_hi(b.y);
  }
}

// Updates a thread's share of the tile at e0 from its loaded inputs and
// stores master, m, v and the rounded bf16 weights.
template <bool kMaster, uint32_t CAP>
__device__ __forceinline__ void update_tile(const StepArgs& p, const SegTable<CAP>& segs, Cursor& c, uint64_t e0,
                                            TileIn& in, float scale, const Hyper& h, uint32_t seed) {
  const uint64_t e1 = e0 + kThreads * kGroup;
  float wd0[kGroup], wd1[kGroup];
  group_decay(c, segs, p, p.goff + e0, wd0);
  group_decay(c, segs, p, p.goff + e1, wd1);

  uint2 q0, q1;
  if constexpr (kMaster) {
    q0 = group_update(in.g0, in.m0, in.v0, in.w0, wd0, scale, h, p.goff + e0, seed);
    q1 = group_update(in.g1, in.m1, in.v1, in.w1, wd1, scale, h, p.goff + e1, seed);
  } else {
    group_update_only(in.g0, in.m0, in.v0, in.w0, wd0, scale, h);
    group_update_only(in.g1, in.m1, in.v1, in.w1, wd1, scale, h);
    sr_pack8(make_float4(in.w0[0], in.w0[1], in.w0[2], in.w0[3]), make_float4(in.w1[0], in.w1[1], in.w1[2], in.w1[3]),
             p.goff + e0, p.goff + e1, seed, q0, q1);
  }

  __stcs(reinterpret_cast<float4*>(p.m + e0), in.m0);
  __stcs(reinterpret_cast<float4*>(p.m + e1), in.m1);
  __stcs(reinterpret_cast<float4*>(p.v + e0), in.v0);
  __stcs(reinterpret_cast<float4*>(p.v + e1), in.v1);
  if (kMaster) {
    __stcs(reinterpret_cast<float4*>(p.master + e0), make_float4(in.w0[0], in.w0[1], in.w0[2], in.w0[3]));
    __stcs(reinterpret_cast<float4*>(p.master + e1), make_float4(in.w1[0], in.w1[1], in.w1[2], in.w1[3]));
  }
  __stcs(reinterpret_cast<uint2*>(p.params + e0), q0);
  __stcs(reinterpret_cast<uint2*>(p.params + e1), q1);
}

// The vector path's tiles for block `block` of `nblocks` (the mapping of a
// grid of nblocks blocks). Requires params/grads 8-B aligned and master/m/v
// 16-B aligned. The first p.head elements (a multiple of 4, below 64) go one
// per thread; then block-iteration k covers tile k of kTile elements from
// element p.head; thread t handles the two 4-element groups at tile offsets
// 4t and 4t + 4*kThreads, so every warp-wide load or store is one contiguous
// 512-B (fp32) or 256-B (bf16) span, which starts on a 128-B line when the
// arrays' starts agree modulo 128 B (the head is chosen for that); the
// ragged tail (< kTile elements) goes one element per thread.
// kHead false compiles the peel away (p.head must then be 0).
template <bool kMaster, bool kHead, uint32_t CAP>
__device__ __forceinline__ void vec_tiles(const StepArgs& p, const SegTable<CAP>& segs, float scale,
                                          const Hyper& h, uint32_t seed, uint32_t block, uint32_t nblocks) {
  const uint64_t head = kHead ? (p.head < p.n ? p.head : p.n) : 0;
  const uint64_t ntiles = (p.n - head) / kTile;
  const uint64_t stride_tail = static_cast<uint64_t>(nblocks) * kThreads;
  const uint64_t lane0 = static_cast<uint64_t>(block) * kThreads + threadIdx.x;
  const uint64_t tail0 = head + ntiles * kTile + lane0;
  uint64_t first = (block < ntiles) ? head + static_cast<uint64_t>(block) * kTile + threadIdx.x * kGroup : tail0;
  if constexpr (kHead) {
    if (lane0 < head) first = lane0;
  }
  if (first >= p.n) first = p.n - 1;
  Cursor c;
  c.s = seg_find(segs, p.nseg, p.goff + first);
  c.end = segs.end[c.s];

  // Head (< 64 elements), one element per thread: indices below every tile's.
  if constexpr (kHead) {
    for (uint64_t i = lane0; i < head; i += stride_tail) elem_update<kMaster>(p, segs, c, i, scale, h, seed);
  }
  for (uint64_t tile = block; tile < ntiles; tile += nblocks) {
    const uint64_t e0 = head + tile * kTile + threadIdx.x * kGroup;
    TileIn in;
    load_tile<kMaster>(p, p.grads, e0, in);
    update_tile<kMaster>(p, segs, c, e0, in, scale, h, seed);
  }
  // Ragged tail (< kTile elements), one element per thread.
  for (uint64_t i = tail0; i < p.n; i += stride_tail) elem_update<kMaster>(p, segs, c, i, scale, h, seed);
}

// ---- tiles staged in shared memory (the TMA path, mp_step.cu) ---------------
// One stage holds a whole 2048-element tile of every input stream, loaded by
// the TMA engine; the update runs on it in place and the TMA engine stores
// the results from it. Byte offsets within a stage:
template <bool kMaster, uint32_t T>
struct TmaStage {
  static_assert(T % 64 == 0, "every stream's tile must span whole 128-B lines");
  static constexpr uint32_t kTileElems = T;
  static constexpr uint32_t kGrads = 0;   // bf16 gradients; with master, the rounded weights go here
  static constexpr uint32_t kW = T * 2;   // the old weights: fp32 master, or the bf16 params in place
  static constexpr uint32_t kM = kW + T * (kMaster ? 4 : 2);
  static constexpr uint32_t kV = kM + T * 4;
  static constexpr uint32_t kBytes = kV + T * 4;  // 14 B per element with master, 12 B without
};

// Updates group g (elements 4g .. 4g + 3) of the tile staged at `sp`, whose
// element 0 is element e0 of the launch: reads the inputs from the stage and
// writes m, v, the master and the rounded weights back into it.
template <bool kMaster, uint32_t T, uint32_t CAP>
__device__ __forceinline__ void stage_group(const StepArgs& p, const SegTable<CAP>& segs, Cursor& c, uint8_t* sp,
                                            uint32_t g, uint64_t e0, float scale, const Hyper& h, uint32_t seed) {
  using L = TmaStage<kMaster, T>;
  const uint64_t gi = p.goff + e0 + 4u * g;
  const uint2 graw = *reinterpret_cast<const uint2*>(sp + L::kGrads + 8u * g);
  float4 m4 = *reinterpret_cast<const float4*>(sp + L::kM + 16u * g);
  float4 v4 = *reinterpret_cast<const float4*>(sp + L::kV + 16u * g);
  float w[kGroup];
  if constexpr (kMaster) {
    const float4 a = *reinterpret_cast<const float4*>(sp + L::kW + 16u * g);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  } else {
    const uint2 a = *reinterpret_cast<const uint2*>(sp + L::kW + 8u * g);
    w[0] = bf16_lo(a.x); w[1] = bf16_hi(a.x); w[2] = bf16_lo(a.y); w[3] = bf16_hi(a.y);
  }
  float wd[kGroup];
  group_decay(c, segs, p, gi, wd);
  const uint2 q = group_update(graw, m4, v4, w, wd, scale, h, gi, seed);
  *reinterpret_cast<float4*>(sp + L::kM + 16u * g) = m4;
  *reinterpret_cast<float4*>(sp + L::kV + 16u * g) = v4;
  if constexpr (kMaster) {
    *reinterpret_cast<float4*>(sp + L::kW + 16u * g) = make_float4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint2*>(sp + L::kGrads + 8u * g) = q;
  } else {
    *reinterpret_cast<uint2*>(sp + L::kW + 8u * g) = q;
  }
}

}  // namespace mpk
