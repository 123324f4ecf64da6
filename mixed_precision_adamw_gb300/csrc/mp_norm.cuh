// mp_norm.cuh — device building blocks of the deterministic gradient norm,
// shared by the two-kernel norm (mp_norm.cu) and the one-launch step for
// small parameter sets (mp_small.cu), which must give identical bits.
//
// llm.c walk-through ch. 04 "Multi-GPU and mixed precision" §4: the train
// step takes the global norm of all gradients with a two-level reduction and
// clips with grad_scale = min(1, 1.0 / grad_norm).
#pragma once

#include <cfloat>
#include <cstdint>

#include "mp_adamw.h"
#include "mp_device.cuh"
#include "mp_internal.h"

namespace mpk {

constexpr int kNormUnroll = 4;  // 16-B loads in flight per thread

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

// Which 8-element vectors norm block `block` of `nblocks` adds, and in what
// order. Long ranges (at least two 256-vector pieces per block) give each
// block one contiguous run of `per` vectors (ceil(nvec / nblocks) rounded up
// to whole 256-vector pieces, so every run starts on a 4 KB boundary of the
// buffer; the last runs end early or are empty): thread t takes vector t of
// each piece, in piece order, so a block's loads are long contiguous spans
// (the TMA-staged kernel fetches a group of pieces with one bulk copy).
// Measured on GB300 (Llama-3-8B gradients): the staged norm took 2.174-2.176
// ms with runs of whole pieces and 2.203-2.206 ms with runs rounded only to
// 128-B lines (better balanced, the same chained step time). Shorter ranges
// interleave the blocks: thread t of block b takes vectors
// b*256 + t + j*nblocks*256. Every kernel of the norm uses this, so the
// host- and device-gradient kernels add the same squares in the same order.
struct NormMap {
  bool contiguous;
  uint64_t first, last;  // contiguous: this block's vectors [first, last)
};

__device__ __forceinline__ NormMap norm_map(uint64_t nvec, uint32_t block, uint32_t nblocks) {
  NormMap m{false, 0, 0};
  const uint64_t stride = static_cast<uint64_t>(nblocks) * kThreads;
  if (nvec < 2 * stride) return m;
  m.contiguous = true;
  const uint64_t per = ((nvec + nblocks - 1) / nblocks + kThreads - 1) / kThreads * kThreads;
  m.first = static_cast<uint64_t>(block) * per < nvec ? static_cast<uint64_t>(block) * per : nvec;
  m.last = m.first + per < nvec ? m.first + per : nvec;
  return m;
}

template <bool kCopy>
__device__ __forceinline__ double norm_block_finish(const uint16_t* __restrict__ grads, uint64_t n, int vec,
                                                    uint16_t* __restrict__ copy_out, uint32_t block,
                                                    uint32_t nblocks, double* sh, float s, float c);

// Partial sum of squares of norm block `block` out of `nblocks`: its vectors
// as norm_map assigns them, then its share of the scalar tail (thread t of
// block b takes elements nvec*8 + b*256 + t + j*nblocks*256). vec: grads (and
// copy_out) 16-B aligned, processed as 8-element vectors plus a scalar tail.
// kCopy: grads may live in page-locked host memory (read over the host link)
// and every element read is also written to copy_out, so the host-to-device
// transfer and the norm are one pass; the arithmetic and its order are the
// same as without the copy. Every thread of the block calls it and receives
// the block's partial.
template <bool kCopy>
__device__ __forceinline__ double norm_block_partial(const uint16_t* __restrict__ grads, uint64_t n, int vec,
                                                     uint16_t* __restrict__ copy_out, uint32_t block,
                                                     uint32_t nblocks, double* sh) {
  const uint4* g4 = reinterpret_cast<const uint4*>(grads);
  uint4* c4 = reinterpret_cast<uint4*>(copy_out);
  const uint64_t nvec = vec ? n / 8 : 0;
  const uint64_t stride = static_cast<uint64_t>(nblocks) * kThreads;
  const uint64_t k0 = static_cast<uint64_t>(block) * kThreads + threadIdx.x;

  float s = 0.0f, c = 0.0f;
  const NormMap map = norm_map(nvec, block, nblocks);
  if (map.contiguous) {
    uint64_t k = map.first + threadIdx.x;
    constexpr uint64_t kStep = kThreads;
    for (; k + (kNormUnroll - 1) * kStep < map.last; k += kNormUnroll * kStep) {
      uint4 w[kNormUnroll];
#pragma unroll
      for (int u = 0; u < kNormUnroll; ++u) w[u] = __ldcs(g4 + k + u * kStep);
      if (kCopy) {
#pragma unroll
        for (int u = 0; u < kNormUnroll; ++u) c4[k + u * kStep] = w[u];
      }
#pragma unroll
      for (int u = 0; u < kNormUnroll; ++u) acc(s, c, sumsq8(w[u]));
    }
    for (; k < map.last; k += kStep) {
      const uint4 w = __ldcs(g4 + k);
      if (kCopy) c4[k] = w;
      acc(s, c, sumsq8(w));
    }
    return norm_block_finish<kCopy>(grads, n, vec, copy_out, block, nblocks, sh, s, c);
  }
  uint64_t k = k0;
  for (; k + (kNormUnroll - 1) * stride < nvec; k += kNormUnroll * stride) {
    uint4 w[kNormUnroll];
#pragma unroll
    for (int u = 0; u < kNormUnroll; ++u) w[u] = __ldcs(g4 + k + u * stride);
    if (kCopy) {
#pragma unroll
      for (int u = 0; u < kNormUnroll; ++u) c4[k + u * stride] = w[u];
    }
#pragma unroll
    for (int u = 0; u < kNormUnroll; ++u) acc(s, c, sumsq8(w[u]));
  }
  for (; k < nvec; k += stride) {
    const uint4 w = __ldcs(g4 + k);
    if (kCopy) c4[k] = w;
    acc(s, c, sumsq8(w));
  }
  return norm_block_finish<kCopy>(grads, n, vec, copy_out, block, nblocks, sh, s, c);
}

// The rest of a norm block's partial after its 8-element vectors have been
// added into (s, c) in the thread's order: the scalar tail, the fixed block
// sum and the fp64 recomputation. Every thread of the block calls it.
template <bool kCopy>
__device__ __forceinline__ double norm_block_finish(const uint16_t* __restrict__ grads, uint64_t n, int vec,
                                                    uint16_t* __restrict__ copy_out, uint32_t block,
                                                    uint32_t nblocks, double* sh, float s, float c) {
  const uint4* g4 = reinterpret_cast<const uint4*>(grads);
  const uint64_t nvec = vec ? n / 8 : 0;
  const uint64_t stride = static_cast<uint64_t>(nblocks) * kThreads;
  const uint64_t k0 = static_cast<uint64_t>(block) * kThreads + threadIdx.x;
  uint64_t k;
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
    const NormMap map = norm_map(nvec, block, nblocks);
    if (map.contiguous) {
      for (k = map.first + threadIdx.x; k < map.last; k += kThreads) d = __dadd_rn(d, dsumsq8(r4[k]));
    } else {
      for (k = k0; k < nvec; k += stride) d = __dadd_rn(d, dsumsq8(r4[k]));
    }
    for (uint64_t i = nvec * 8 + k0; i < n; i += stride) {
      const double x = bf16_to_f32(r1[i]);
      d = __dadd_rn(d, __dmul_rn(x, x));
    }
    S = block_sum(d, sh);
  }
  return S;
}

// Level 2: the sum of the nblocks partials in a fixed order (thread t adds
// partials t, t + 256, ..., then the fixed block tree); every thread of the
// block calls it and receives the total. partial(i) returns partial i.
template <typename PartialAt>
__device__ __forceinline__ double norm_total(PartialAt partial, int nblocks, double* sh) {
  double d = 0.0;
  for (int i = threadIdx.x; i < nblocks; i += kThreads) d = __dadd_rn(d, partial(i));
  return block_sum(d, sh);
}

// The norm and clip scale from the total sum of squares S.
__device__ __forceinline__ void norm_and_scale(double S, float clip, float& norm, float& scale) {
  norm = __double2float_rn(__dsqrt_rn(S));
  if (!isfinite(norm)) {
    scale = __int_as_float(0x7FC00000);  // NaN: the step refuses to run
  } else {
    const float q = __fdiv_rn(clip, norm);  // norm == 0 gives +Inf -> 1
    scale = q < 1.0f ? q : 1.0f;
  }
}

// The step a device step counter would take next, from the state as it is
// now: t, its seed and bias corrections, and the learning rate. ok is false
// when the step cannot be taken: a negative or saturated count, or a t beyond
// a bias table whose last entry is not (1, 1).
struct ClockStep {
  int32_t t;
  uint32_t seed;
  float bc1, bc2, lr;
  bool ok;
};

__device__ __forceinline__ ClockStep next_clock_step(const StepClock& c) {
  const mp_step_state_t* st = c.state;
  ClockStep s{0, 0u, 0.0f, 0.0f, st->lr, false};
  const int32_t t0 = st->t;
  if (t0 < 0 || t0 == 0x7FFFFFFF) return s;
  s.t = t0 + 1;
  const int64_t last = c.bias_len - 1;
  const int64_t k = (static_cast<int64_t>(s.t) - 1 < last) ? static_cast<int64_t>(s.t) - 1 : last;
  s.bc1 = c.bias[2 * k];
  s.bc2 = c.bias[2 * k + 1];
  s.seed = st->seed_base + static_cast<uint32_t>(s.t);
  s.ok = !(static_cast<int64_t>(s.t) - 1 > last && !(s.bc1 == 1.0f && s.bc2 == 1.0f));
  return s;
}

// Records a taken step in the state (one thread).
__device__ __forceinline__ void commit_clock_step(const StepClock& c, const ClockStep& s) {
  mp_step_state_t* st = c.state;
  st->t = s.t;
  st->seed = s.seed;
  st->bc1 = s.bc1;
  st->bc2 = s.bc2;
}

// Advances the device step counter (one thread); false, leaving the state
// untouched, when the step cannot be taken.
__device__ __forceinline__ bool advance_clock(const StepClock& c) {
  const ClockStep s = next_clock_step(c);
  if (s.ok) commit_clock_step(c, s);
  return s.ok;
}

}  // namespace mpk
