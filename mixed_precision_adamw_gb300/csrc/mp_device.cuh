// mp_device.cuh — device-side building blocks of the optimizer step.
//
// Sources (web pages, by title and section):
//   llm.c walk-through ch. 04 "Multi-GPU and mixed precision": §2.2 AdamW
//   kernel (per-parameter update, two-FMA lerp), §2.3 stochastic rounding
//   with SquirrelNoise5 draws.
//
// All floating-point operations are written as explicit round-to-nearest
// intrinsics so that no FMA contraction or fast-math rewrite can change a
// result: the update is bit-reproducible and matches its written definition.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mpk {

constexpr int kThreads = 256;          // threads per block in every kernel
constexpr int kGroup = 4;              // consecutive elements per fp32 16-B vector
constexpr int kTile = kThreads * kGroup * 2;  // elements per block-iteration (two groups per thread)

// ---- programmatic dependent launch ----------------------------------------
// Every kernel is launched with programmatic stream serialisation allowed, so
// the GPU may schedule it while the previous kernel in the stream is still
// finishing. griddepcontrol.wait blocks until that previous grid has completed
// and its memory writes are visible; it comes before any global memory access.
// launch_dependents then lets the next kernel in the stream be scheduled early
// (it, too, waits before touching memory).
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- rounding randomness ---------------------------------------------------
// SquirrelNoise5 (Squirrel Eiserloh's published counter-based noise hash) in
// its 2D form, evaluated at x = low word, y = high word of the 64-bit global
// element index. A pure function of (index, seed): independent of the grid.
constexpr uint32_t kNoisePrime = 198491317u;  // folds y into x (the 2D entry)

// 2D fold of a global index into the 1D noise position.
__device__ __forceinline__ uint32_t noise_pos(uint64_t k) {
  return static_cast<uint32_t>(k) + kNoisePrime * static_cast<uint32_t>(k >> 32);
}

constexpr uint32_t kNoiseMul1 = 0xD2A80A3Fu;   // the first round's multiplier

// The first SquirrelNoise5 round: pos * C1 + seed.
__device__ __forceinline__ uint32_t noise_first(uint32_t pos, uint32_t seed) { return pos * kNoiseMul1 + seed; }

// Every round after the first, except the final xor-shift by 17.
__device__ __forceinline__ uint32_t noise_rest(uint32_t h) {
  h ^= h >> 9;
  h += 0xA884F197u;
  h ^= h >> 11;
  h *= 0x6C736F4Bu;
  h ^= h >> 13;
  h += 0xB79F3ABBu;
  h ^= h >> 15;
  h *= 0x1B56C4F5u;
  return h;
}

// Every SquirrelNoise5 round except the final xor-shift by 17.
__device__ __forceinline__ uint32_t noise_rounds(uint32_t pos, uint32_t seed) {
  return noise_rest(noise_first(pos, seed));
}

__device__ __forceinline__ uint32_t noise_u32(uint64_t k, uint32_t seed) {
  const uint32_t h = noise_rounds(noise_pos(k), seed);
  return h ^ (h >> 17);
}

// 0xFFFF minus the 16-bit draw (the low half of the noise), i.e. ~draw & 0xFFFF,
// from the first round's value h1 = noise_first(pos, seed).
__device__ __forceinline__ uint32_t draw16_complement_h1(uint32_t h1) {
  const uint32_t h = noise_rest(h1);
  return ~(h ^ (h >> 17)) & 0xFFFFu;
}

__device__ __forceinline__ uint32_t draw16_complement(uint32_t pos, uint32_t seed) {
  return draw16_complement_h1(noise_first(pos, seed));
}

// Noise positions of the 4 consecutive indices k0 .. k0+3 from one fold:
// noise_pos(k0 + j) = noise_pos(k0) + j, plus the prime once if the low word
// wrapped past 2^32 between k0 and k0 + j (the high word then grew by one).
// Branch-free, so the unrolled update is not duplicated per case.
__device__ __forceinline__ void noise_pos4(uint64_t k0, uint32_t (&pos)[4]) {
  const uint32_t lo = static_cast<uint32_t>(k0);
  const uint32_t p0 = noise_pos(k0);
#pragma unroll
  for (int j = 0; j < 4; ++j) pos[j] = p0 + j + (lo > 0xFFFFFFFFu - j ? kNoisePrime : 0u);
}

// First-round values h1[j] = noise_first(noise_pos(k0 + j), seed) of the 4
// consecutive indices k0 .. k0+3. When their low words do not wrap past 2^32
// (all but one group in 2^30), noise_pos(k0 + j) = noise_pos(k0) + j, so
// h1[j] = h1[0] + j * C1 (mod 2^32): one multiply-add for the group and one
// constant addition per further element, instead of a position, a wrap test
// and a multiply-add per element. The rare wrapping group takes noise_pos4.
__device__ __forceinline__ void noise_first4(uint64_t k0, uint32_t seed, uint32_t (&h1)[4]) {
  if (static_cast<uint32_t>(k0) <= 0xFFFFFFFCu) {
    const uint32_t b = noise_first(noise_pos(k0), seed);
#pragma unroll
    for (int j = 0; j < 4; ++j) h1[j] = b + static_cast<uint32_t>(j) * kNoiseMul1;
  } else {
    uint32_t pos[4];
    noise_pos4(k0, pos);
#pragma unroll
    for (int j = 0; j < 4; ++j) h1[j] = noise_first(pos[j], seed);
  }
}

// True when none of the 8 values is NaN: their sum is then not NaN unless
// infinities of both signs meet, which only sends such a group to the path
// that checks every element. The additions run on the FMA pipe, which the
// rounding kernels leave mostly idle, instead of a compare and a select per
// element on the integer pipe.
__device__ __forceinline__ bool none_nan8(const float4& a, const float4& b) {
  const float s = __fadd_rn(__fadd_rn(__fadd_rn(a.x, a.y), __fadd_rn(a.z, a.w)),
                            __fadd_rn(__fadd_rn(b.x, b.y), __fadd_rn(b.z, b.w)));
  return s == s;
}

// ---- stochastic rounding fp32 -> bf16 -------------------------------------
// Keep the top half of the fp32 pattern and add one (the bf16 neighbour away
// from zero) when the discarded low half exceeds a uniform 16-bit draw r, so
// the probability of rounding away from zero is lo16 / 65536. With
// c = 0xFFFF - r, the carry out of lo16 + c is exactly [lo16 > r], so the
// result is the high half of b + c (no non-NaN pattern overflows: the largest
// is -Inf, 0xFF800000). NaN becomes the canonical quiet NaN (truncation could
// otherwise yield an infinity).
__device__ __forceinline__ uint32_t sr_bf16_c(float x, uint32_t draw_complement) {
  const uint32_t b = __float_as_uint(x);
  const uint32_t r = (b + draw_complement) >> 16;
  return (x != x) ? 0x7FC0u : r;  // x != x: NaN (a float compare keeps the integer pipe free)
}

// The same rounding, left in the high half of a 32-bit word (the low half is
// left over): SR(x) = sr_bf16_hi(x, c) >> 16. Two such words pack into one
// word of two bf16 with a single byte permute (pack_hi16), so the vector
// paths spend no shifts on the results.
__device__ __forceinline__ uint32_t sr_bf16_hi(float x, uint32_t draw_complement) {
  const uint32_t b = __float_as_uint(x);
  return (x != x) ? 0x7FC00000u : b + draw_complement;
}

// (hi16(lo_word)) | (hi16(hi_word) << 16): bytes 2, 3 of lo_word, then bytes
// 2, 3 of hi_word.
__device__ __forceinline__ uint32_t pack_hi16(uint32_t lo_word, uint32_t hi_word) {
  return __byte_perm(lo_word, hi_word, 0x7632);
}

// Stochastic rounding of a thread's two 4-element groups a (global indices
// k0 .. k0+3) and b (k1 .. k1+3), packed as bf16 pairs. Without NaN among
// the 8 values (none_nan8) each result is the high half of b + c, with no
// per-element NaN select; otherwise sr_bf16_hi per element.
__device__ __forceinline__ void sr_pack8(const float4& a, const float4& b, uint64_t k0, uint64_t k1, uint32_t seed,
                                         uint2& qa, uint2& qb) {
  uint32_t ha[4], hb[4];
  noise_first4(k0, seed, ha);
  noise_first4(k1, seed, hb);
  if (none_nan8(a, b)) {
    qa.x = pack_hi16(__float_as_uint(a.x) + draw16_complement_h1(ha[0]),
                     __float_as_uint(a.y) + draw16_complement_h1(ha[1]));
    qa.y = pack_hi16(__float_as_uint(a.z) + draw16_complement_h1(ha[2]),
                     __float_as_uint(a.w) + draw16_complement_h1(ha[3]));
    qb.x = pack_hi16(__float_as_uint(b.x) + draw16_complement_h1(hb[0]),
                     __float_as_uint(b.y) + draw16_complement_h1(hb[1]));
    qb.y = pack_hi16(__float_as_uint(b.z) + draw16_complement_h1(hb[2]),
                     __float_as_uint(b.w) + draw16_complement_h1(hb[3]));
  } else {
    qa.x = pack_hi16(sr_bf16_hi(a.x, draw16_complement_h1(ha[0])), sr_bf16_hi(a.y, draw16_complement_h1(ha[1])));
    qa.y = pack_hi16(sr_bf16_hi(a.z, draw16_complement_h1(ha[2])), sr_bf16_hi(a.w, draw16_complement_h1(ha[3])));
    qb.x = pack_hi16(sr_bf16_hi(b.x, draw16_complement_h1(hb[0])), sr_bf16_hi(b.y, draw16_complement_h1(hb[1])));
    qb.y = pack_hi16(sr_bf16_hi(b.z, draw16_complement_h1(hb[2])), sr_bf16_hi(b.w, draw16_complement_h1(hb[3])));
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

// ---- the per-element AdamW update ------------------------------------------
struct Hyper {
  float lr, beta1, beta2, eps, wd, bc1, bc2;
};

// lerp(start, end, w) = w * end + (start - w * start): two FMAs.
__device__ __forceinline__ float lerp2(float start, float end, float w) {
  return __fmaf_rn(w, end, __fmaf_rn(-w, start, start));
}

// Updates m and v in place and returns the new fp32 weight.
//   g = scale * grad;  m = lerp(g, m, b1);  v = lerp(g*g, v, b2)
//   p = old - lr * ( (m/bc1) / (sqrt(v/bc2) + eps) + wd_e * old )
__device__ __forceinline__ float adamw_update(float grad, float& m, float& v, float old,
                                              float wd_e, float scale, const Hyper& h) {
  const float g = __fmul_rn(scale, grad);
  m = lerp2(g, m, h.beta1);
  const float gg = __fmul_rn(g, g);
  v = lerp2(gg, v, h.beta2);
  const float m_hat = __fdiv_rn(m, h.bc1);
  const float v_hat = __fdiv_rn(v, h.bc2);
  const float denom = __fadd_rn(__fsqrt_rn(v_hat), h.eps);
  const float update = __fadd_rn(__fdiv_rn(m_hat, denom), __fmul_rn(wd_e, old));
  return __fsub_rn(old, __fmul_rn(h.lr, update));
}

}  // namespace mpk
