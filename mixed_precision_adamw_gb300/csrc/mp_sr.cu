// mp_sr.cu — standalone stochastic rounding fp32 -> bf16 and fp32 -> fp16,
// accumulation into bf16 with stochastic rounding, and the rounding
// randomness itself.
//
// llm.c walk-through ch. 04 "Multi-GPU and mixed precision" §2.3 (the rule)
// and §5.2 (bf16 weights are rebuilt from the fp32 master with the saved
// rounding randomness, so a resumed run is bit-identical). Because the draw is
// keyed on the global element index, the rebuild needs no launch-geometry
// alignment: any grid gives the same bits. 6 B of HBM traffic per element;
// at that ratio the draw's integer work (about 19 operations per element)
// keeps the integer ALU pipe busy, so the register kernels run a little below
// the memory bound; long aligned ranges of the bf16 rounding and of the
// accumulation take TMA-staged kernels (below), which hide the memory latency
// from the warps. The same section has the rounding write the encoder's
// embedding gradients: a bf16 gradient plus an fp32 contribution, rounded
// back (8 B per element).
#include <atomic>

#include "mp_device.cuh"
#include "mp_internal.h"
#include "mp_tma.cuh"

namespace mpk {
namespace {

constexpr int kSrBlocksPerSm = 8;

// Stochastic rounding fp32 -> fp16: the bf16 rule on fp16's grid. Between
// the fp16 neighbour toward zero and the next one away from zero, round away
// when the discarded fraction of one fp16 step, cut to 16 bits, exceeds the
// 16-bit draw. As for bf16, the work is one 32-bit word v whose high half is
// the truncated fp16 pattern and whose low half is that 16-bit fraction; then
// hi16(v + 0xFFFF - draw) carries exactly when the fraction exceeds the draw,
// and the carry runs into the exponent (0x03FF + 1 is the smallest normal,
// 0x7BFF + 1 infinity). Two candidate words, of which v is the smaller:
//   v_normal: the pattern of |x| clamped to [2^-14, 65536], rebiased from
//     127 to 15 and shifted left by 3 (pattern * 8 + 0x40000000 modulo
//     2^32), so the 10 kept mantissa bits end at bit 16 and the 13 dropped
//     ones fill bits 15..3. Exact for 2^-14 <= |x| < 65536; 0x7C000000
//     (infinity, no carry possible) from 65536 up; 2^26 below 2^-14.
//   v_sub: floor(|x| * 2^40) (the product is exact; the conversion truncates
//     and saturates at 2^32 - 1), fp16 subnormal steps of 2^-24 in the high
//     half and the fraction in the low. Exact below 2^-14, where it is below
//     2^26; from 2^-14 up it is never below v_normal (the linear scale grows
//     at least as fast as the exponent-and-mantissa one, and they meet at
//     2^-14).
// NaN gives the canonical quiet NaN 0x7E00; otherwise the sign is kept.
// The conversion and the multiplies run on the FMA and conversion pipes,
// which this integer-heavy kernel leaves mostly idle.
// Returns the fp16 pattern in the high half of the word.
__device__ __forceinline__ uint32_t sr_fp16_hi(float x, uint32_t draw_complement) {
  const float a = fabsf(x);
  const uint32_t v_normal = __float_as_uint(fminf(fmaxf(a, 0x1p-14f), 65536.0f)) * 8u + 0x40000000u;
  const uint32_t v_sub = __float2uint_rz(__fmul_rn(a, 0x1p40f));
  const uint32_t w = (min(v_normal, v_sub) + draw_complement) | (__float_as_uint(x) & 0x80000000u);
  return x != x ? 0x7E000000u : w;
}

// True when 2^-14 <= |x| < 65536 (fp16's normal range), where sr_fp16_hi
// reduces to sr_fp16_hi_normal. Doubling the pattern drops the sign bit; the
// range is then [0x71000000, 0x8F000000), tested with one unsigned compare.
__device__ __forceinline__ bool fp16_normal_range(float x) {
  return __float_as_uint(x) * 2u - 0x71000000u < 0x1E000000u;
}

// sr_fp16_hi for x in fp16's normal range: (|x| pattern - 0x38000000) << 3
// is |x| pattern * 8 + 0x40000000 modulo 2^32, and shifting the pattern left
// by 3 drops the sign bit, so no mask is needed.
__device__ __forceinline__ uint32_t sr_fp16_hi_normal(float x, uint32_t draw_complement) {
  const uint32_t b = __float_as_uint(x);
  return ((b << 3) + 0x40000000u + draw_complement) | (b & 0x80000000u);
}

// Four consecutive elements with first-round noise values h1[0..3], packed
// as fp16.
template <bool kNormalOnly>
__device__ __forceinline__ uint2 sr_fp16_pack4(const float4& x, const uint32_t (&h1)[kGroup]) {
  auto r = [&](float v, uint32_t h) {
    return kNormalOnly ? sr_fp16_hi_normal(v, draw16_complement_h1(h)) : sr_fp16_hi(v, draw16_complement_h1(h));
  };
  uint2 q;
  q.x = pack_hi16(r(x.x, h1[0]), r(x.y, h1[1]));
  q.y = pack_hi16(r(x.z, h1[2]), r(x.w, h1[3]));
  return q;
}

// Vector path: in 16-B aligned, out 8-B aligned. Same tiling as the step:
// thread t converts the 4-element groups at tile offsets 4t and 4t + 1024.
__global__ void __launch_bounds__(kThreads, kSrBlocksPerSm)
sr_vec_kernel(uint16_t* __restrict__ out, const float* __restrict__ in, uint64_t goff, uint64_t n, uint32_t seed) {
  pdl_enter();
  const uint64_t ntiles = n / kTile;
  for (uint64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const uint64_t e0 = tile * kTile + threadIdx.x * kGroup;
    const uint64_t e1 = e0 + kThreads * kGroup;
    const float4 a = __ldcs(reinterpret_cast<const float4*>(in + e0));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(in + e1));
    uint2 qa, qb;
    sr_pack8(a, b, goff + e0, goff + e1, seed, qa, qb);
    __stcs(reinterpret_cast<uint2*>(out + e0), qa);
    __stcs(reinterpret_cast<uint2*>(out + e1), qb);
  }
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
  for (uint64_t i = ntiles * kTile + static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n; i += stride)
    out[i] = static_cast<uint16_t>(sr_bf16_c(in[i], draw16_complement(noise_pos(goff + i), seed)));
}

__global__ void __launch_bounds__(kThreads)
sr_scalar_kernel(uint16_t* __restrict__ out, const float* __restrict__ in, uint64_t goff, uint64_t n, uint32_t seed) {
  pdl_enter();
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n; i += stride)
    out[i] = static_cast<uint16_t>(sr_bf16_c(in[i], draw16_complement(noise_pos(goff + i), seed)));
}

// out[i] = fp16 stochastic rounding of in[i] (sr_fp16_hi), with the draws of
// the bf16 rounding. Vector path: in 16-B aligned, out 8-B aligned.
__global__ void __launch_bounds__(kThreads, kSrBlocksPerSm)
sr_fp16_vec_kernel(uint16_t* __restrict__ out, const float* __restrict__ in, uint64_t goff, uint64_t n,
                   uint32_t seed) {
  pdl_enter();
  const uint64_t ntiles = n / kTile;
  for (uint64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const uint64_t e0 = tile * kTile + threadIdx.x * kGroup;
    const uint64_t e1 = e0 + kThreads * kGroup;
    const float4 a = __ldcs(reinterpret_cast<const float4*>(in + e0));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(in + e1));
    uint32_t pa[kGroup], pb[kGroup];
    noise_first4(goff + e0, seed, pa);
    noise_first4(goff + e1, seed, pb);
    // Per group set (a: groups 4t, b: groups 4t + 1024): a warp whose 128
    // elements all lie in fp16's normal range takes the short form; the
    // vote keeps the warp converged.
    const bool na = fp16_normal_range(a.x) & fp16_normal_range(a.y) & fp16_normal_range(a.z) & fp16_normal_range(a.w);
    const bool nb = fp16_normal_range(b.x) & fp16_normal_range(b.y) & fp16_normal_range(b.z) & fp16_normal_range(b.w);
    const uint2 qa = __all_sync(0xFFFFFFFFu, na) ? sr_fp16_pack4<true>(a, pa) : sr_fp16_pack4<false>(a, pa);
    const uint2 qb = __all_sync(0xFFFFFFFFu, nb) ? sr_fp16_pack4<true>(b, pb) : sr_fp16_pack4<false>(b, pb);
    __stcs(reinterpret_cast<uint2*>(out + e0), qa);
    __stcs(reinterpret_cast<uint2*>(out + e1), qb);
  }
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
  for (uint64_t i = ntiles * kTile + static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n; i += stride)
    out[i] = static_cast<uint16_t>(sr_fp16_hi(in[i], draw16_complement(noise_pos(goff + i), seed)) >> 16);
}

__global__ void __launch_bounds__(kThreads)
sr_fp16_scalar_kernel(uint16_t* __restrict__ out, const float* __restrict__ in, uint64_t goff, uint64_t n,
                      uint32_t seed) {
  pdl_enter();
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n; i += stride)
    out[i] = static_cast<uint16_t>(sr_fp16_hi(in[i], draw16_complement(noise_pos(goff + i), seed)) >> 16);
}

// acc[i] = SR((float)acc[i] + delta[i], goff + i, seed), in place. Vector
// path: acc 8-B aligned, delta 16-B aligned; the step's tiling.
__global__ void __launch_bounds__(kThreads, kSrBlocksPerSm)
accumulate_vec_kernel(uint16_t* __restrict__ acc, const float* __restrict__ delta, uint64_t goff, uint64_t n,
                      uint32_t seed) {
  pdl_enter();
  const uint64_t ntiles = n / kTile;
  for (uint64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const uint64_t e0 = tile * kTile + threadIdx.x * kGroup;
    const uint64_t e1 = e0 + kThreads * kGroup;
    const uint2 a0 = __ldcs(reinterpret_cast<const uint2*>(acc + e0));
    const uint2 a1 = __ldcs(reinterpret_cast<const uint2*>(acc + e1));
    const float4 d0 = __ldcs(reinterpret_cast<const float4*>(delta + e0));
    const float4 d1 = __ldcs(reinterpret_cast<const float4*>(delta + e1));
    const float4 s0 = make_float4(__fadd_rn(bf16_lo(a0.x), d0.x), __fadd_rn(bf16_hi(a0.x), d0.y),
                                  __fadd_rn(bf16_lo(a0.y), d0.z), __fadd_rn(bf16_hi(a0.y), d0.w));
    const float4 s1 = make_float4(__fadd_rn(bf16_lo(a1.x), d1.x), __fadd_rn(bf16_hi(a1.x), d1.y),
                                  __fadd_rn(bf16_lo(a1.y), d1.z), __fadd_rn(bf16_hi(a1.y), d1.w));
    uint2 q0, q1;
    sr_pack8(s0, s1, goff + e0, goff + e1, seed, q0, q1);
    __stcs(reinterpret_cast<uint2*>(acc + e0), q0);
    __stcs(reinterpret_cast<uint2*>(acc + e1), q1);
  }
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
  for (uint64_t i = ntiles * kTile + static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n; i += stride)
    acc[i] = static_cast<uint16_t>(
        sr_bf16_c(__fadd_rn(bf16_to_f32(acc[i]), delta[i]), draw16_complement(noise_pos(goff + i), seed)));
}

__global__ void __launch_bounds__(kThreads)
accumulate_scalar_kernel(uint16_t* __restrict__ acc, const float* __restrict__ delta, uint64_t goff, uint64_t n,
                         uint32_t seed) {
  pdl_enter();
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n; i += stride)
    acc[i] = static_cast<uint16_t>(
        sr_bf16_c(__fadd_rn(bf16_to_f32(acc[i]), delta[i]), draw16_complement(noise_pos(goff + i), seed)));
}

// ---- TMA-staged rounding (long aligned ranges) --------------------------------
// The bf16 rounding and accumulate-and-round kernels above on tiles that the
// TMA engine stages in shared memory, as the step kernel's TMA path does: one
// block per SM; thread 0 has whole tiles of the inputs loaded by bulk copies
// into a ring of stages and, once the consumer warps have rounded a tile, the
// output stored by bulk copies. Consumer thread c rounds the 4-element groups
// c and c + consumers of a tile with the code of the register kernels (the
// same draws and bits). Every wait gives up after one second; nothing then
// reports it, but the outputs of the tiles not stored stay as they were.
// Measured on GB300 (201M elements, interleaved builds): bf16 rounding 6.44
// TB/s at 24 consumer warps x 6 stages (16 x 6: 6.03, 28 x 5: 6.42, 16 x 4:
// 5.35) against 6.25 for sr_vec_kernel; accumulate-and-round 6.83 at 16 x 6
// (12 x 8: 6.85, 24 x 4: 6.72, 8 x 4: 4.82) against 6.26-6.32 for
// accumulate_vec_kernel. The fp16 rounding stays on its register kernel:
// bound by the integer pipe, it ran 5.53-5.58 staged against 5.58-5.60.
enum class RoundKind { kBf16, kAccumulate };

template <RoundKind K>
struct RoundTma {
  static constexpr int kConsumerWarps = K == RoundKind::kAccumulate ? 16 : 24;
  static constexpr uint32_t kStages = 6;
  // Ranges shorter than this many tiles per SM keep the register kernel: the
  // pipeline's fill and drain cost more than the staging saves. Measured on
  // GB300 against the register kernels (3 interleaved runs each): bf16
  // rounding -17 % at 16.8M elements (18 tiles per SM), -10 % at 33.6M,
  // -1.5 % at 67.1M (72), +3 % at 201M (215); accumulate -16 % at 16.8M
  // (27), -13 % at 33.6M (54), +2.3 % at 67.1M (108), +8 % at 201M.
  static constexpr uint64_t kMinTilesPerSm = K == RoundKind::kAccumulate ? 80 : 128;
  static constexpr int kConsumers = 32 * kConsumerWarps;
  static constexpr int kThreads = 32 + kConsumers;
  static constexpr uint32_t kTileElems = static_cast<uint32_t>(kConsumers) * 2 * kGroup;
  // Stage layout. Rounding: the fp32 inputs, then the bf16 outputs.
  // Accumulate: the bf16 accumulators (rounded in place), then the fp32
  // contributions.
  static constexpr uint32_t kIn = K == RoundKind::kAccumulate ? kTileElems * 2 : 0;      // fp32
  static constexpr uint32_t kOut = K == RoundKind::kAccumulate ? 0 : kTileElems * 4;     // 16-bit
  static constexpr uint32_t kBytes = kTileElems * 6;
  // bytes the loads of one tile bring (the barrier's expected count)
  static constexpr uint32_t kLoadBytes = K == RoundKind::kAccumulate ? kTileElems * 6 : kTileElems * 4;
  static constexpr size_t kSmemBytes = kStages * kBytes + 16 * kStages;
};

template <RoundKind K>
__global__ void __launch_bounds__(RoundTma<K>::kThreads, 1)
round_tma_kernel(uint16_t* __restrict__ out, const float* __restrict__ in, uint64_t goff, uint64_t n,
                 uint32_t seed) {
  pdl_enter();
  using C = RoundTma<K>;
  constexpr uint32_t S = C::kStages, T = C::kTileElems;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t base = smem_u32(smem), full = base + S * C::kBytes, done = full + 8 * S;
  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < S; ++i) {
      mbar_init(full + 8 * i, 1);
      mbar_init(done + 8 * i, C::kConsumerWarps);
    }
    mbar_init_fence();
  }
  __syncthreads();
  const uint64_t ntiles = n / T;
  const uint64_t mine = blockIdx.x < ntiles ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  auto elem = [&](uint64_t k) { return (blockIdx.x + k * gridDim.x) * static_cast<uint64_t>(T); };

  if (threadIdx.x < 32) {  // the producer
    if (threadIdx.x != 0) return;
    const uint64_t pol = l2_evict_first();
    auto load = [&](uint64_t k) {
      const uint32_t st = static_cast<uint32_t>(k % S), bar = full + 8 * st, sp = base + st * C::kBytes;
      const uint64_t e = elem(k);
      mbar_expect_tx(bar, C::kLoadBytes);
      if constexpr (K == RoundKind::kAccumulate) bulk_load(sp, out + e, T * 2, bar, pol);
      bulk_load(sp + C::kIn, in + e, T * 4, bar, pol);
    };
    uint64_t issued = 0, k = 0;
    for (; issued < mine && issued + 1 < S; ++issued) load(issued);
    bool ok = true;
    for (; k < mine; ++k) {
      const uint32_t st = static_cast<uint32_t>(k % S);
      if (!mbar_wait(done + 8 * st, static_cast<uint32_t>((k / S) & 1))) {
        ok = false;
        break;
      }
      bulk_store(out + elem(k), base + st * C::kBytes + C::kOut, T * 2, pol);
      bulk_commit();
      if (issued < mine) {
        bulk_wait_read<1>();
        load(issued++);
      }
    }
    if (!ok)
      for (uint64_t j = k; j < issued; ++j)
        mbar_wait(full + 8 * static_cast<uint32_t>(j % S), static_cast<uint32_t>((j / S) & 1));
    bulk_wait_all();
    return;
  }

  const uint32_t ci = threadIdx.x - 32;
  for (uint64_t k = 0; k < mine; ++k) {
    const uint32_t st = static_cast<uint32_t>(k % S);
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(full + 8 * st, static_cast<uint32_t>((k / S) & 1)))) break;
    uint8_t* sp = smem + st * C::kBytes;
    const uint64_t e0 = goff + elem(k) + 4u * ci, e1 = e0 + 4u * C::kConsumers;
    const float4 a = *reinterpret_cast<const float4*>(sp + C::kIn + 16u * ci);
    const float4 b = *reinterpret_cast<const float4*>(sp + C::kIn + 16u * (ci + C::kConsumers));
    uint2 qa, qb;
    if constexpr (K == RoundKind::kBf16) {
      sr_pack8(a, b, e0, e1, seed, qa, qb);
    } else {
      const uint2 a0 = *reinterpret_cast<const uint2*>(sp + 8u * ci);
      const uint2 a1 = *reinterpret_cast<const uint2*>(sp + 8u * (ci + C::kConsumers));
      const float4 s0 = make_float4(__fadd_rn(bf16_lo(a0.x), a.x), __fadd_rn(bf16_hi(a0.x), a.y),
                                    __fadd_rn(bf16_lo(a0.y), a.z), __fadd_rn(bf16_hi(a0.y), a.w));
      const float4 s1 = make_float4(__fadd_rn(bf16_lo(a1.x), b.x), __fadd_rn(bf16_hi(a1.x), b.y),
                                    __fadd_rn(bf16_lo(a1.y), b.z), __fadd_rn(bf16_hi(a1.y), b.w));
      sr_pack8(s0, s1, e0, e1, seed, qa, qb);
    }
    *reinterpret_cast<uint2*>(sp + C::kOut + 8u * ci) = qa;
    *reinterpret_cast<uint2*>(sp + C::kOut + 8u * (ci + C::kConsumers)) = qb;
    fence_to_bulk();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(done + 8 * st);
  }
  // ragged tail (< T elements), one element per thread
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * C::kConsumers;
  for (uint64_t i = ntiles * T + static_cast<uint64_t>(blockIdx.x) * C::kConsumers + ci; i < n; i += stride) {
    const uint32_t d = draw16_complement(noise_pos(goff + i), seed);
    if constexpr (K == RoundKind::kBf16) out[i] = static_cast<uint16_t>(sr_bf16_c(in[i], d));
    else out[i] = static_cast<uint16_t>(sr_bf16_c(__fadd_rn(bf16_to_f32(out[i]), in[i]), d));
  }
}

// Launches round_tma_kernel<K> when the range holds at least kMinTilesPerSm
// tiles per SM and both arrays are 16-B aligned (so every tile starts
// aligned); false when it does not apply.
template <RoundKind K>
bool launch_round_tma(uint16_t* out, const float* in, uint64_t goff, uint64_t n, uint32_t seed,
                      const DeviceInfo& dev, cudaStream_t stream, cudaError_t* err) {
  using C = RoundTma<K>;
  if (reinterpret_cast<uintptr_t>(out) % 16 || reinterpret_cast<uintptr_t>(in) % 16 ||
      n / C::kTileElems < C::kMinTilesPerSm * static_cast<uint64_t>(dev.sms))
    return false;
  static std::atomic<bool> smem_set[64];
  if (dev.device < 0 || dev.device >= 64 || !smem_set[dev.device].load(std::memory_order_relaxed)) {
    const cudaError_t e = cudaFuncSetAttribute(round_tma_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(C::kSmemBytes));
    if (e != cudaSuccess) {
      *err = e;
      return true;
    }
    if (dev.device >= 0 && dev.device < 64) smem_set[dev.device].store(true, std::memory_order_relaxed);
  }
  *err = launch_pdl_smem(round_tma_kernel<K>, static_cast<unsigned>(dev.sms), C::kThreads, C::kSmemBytes, stream,
                         out, in, goff, n, seed);
  return true;
}

__global__ void __launch_bounds__(kThreads)
noise_kernel(uint32_t* __restrict__ out, uint64_t first, uint64_t n, uint32_t seed) {
  pdl_enter();
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kThreads;
  for (uint64_t i = static_cast<uint64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n; i += stride)
    out[i] = noise_u32(first + i, seed);
}

unsigned grid_for(uint64_t units, const DeviceInfo& dev) {
  uint64_t blocks = (units + kThreads - 1) / kThreads;
  const uint64_t cap = static_cast<uint64_t>(dev.sms) * kSrBlocksPerSm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<unsigned>(blocks);
}

}  // namespace

cudaError_t launch_sr(uint16_t* out, const float* in, uint64_t goff, uint64_t n, uint32_t seed, bool vec,
                      const DeviceInfo& dev, cudaStream_t stream) {
  cudaError_t e;
  if (vec && launch_round_tma<RoundKind::kBf16>(out, in, goff, n, seed, dev, stream, &e)) return e;
  if (vec) {
    const uint64_t ntiles = n / kTile;
    const unsigned blocks = ntiles ? grid_for(ntiles * kThreads, dev) : grid_for(n, dev);
    return launch_pdl(sr_vec_kernel, blocks, kThreads, stream, out, in, goff, n, seed);
  }
  return launch_pdl(sr_scalar_kernel, grid_for(n, dev), kThreads, stream, out, in, goff, n, seed);
}

cudaError_t launch_sr_fp16(uint16_t* out, const float* in, uint64_t goff, uint64_t n, uint32_t seed, bool vec,
                           const DeviceInfo& dev, cudaStream_t stream) {
  if (vec) {
    const uint64_t ntiles = n / kTile;
    const unsigned blocks = ntiles ? grid_for(ntiles * kThreads, dev) : grid_for(n, dev);
    return launch_pdl(sr_fp16_vec_kernel, blocks, kThreads, stream, out, in, goff, n, seed);
  }
  return launch_pdl(sr_fp16_scalar_kernel, grid_for(n, dev), kThreads, stream, out, in, goff, n, seed);
}

cudaError_t launch_accumulate_sr(uint16_t* acc, const float* delta, uint64_t goff, uint64_t n, uint32_t seed,
                                 bool vec, const DeviceInfo& dev, cudaStream_t stream) {
  cudaError_t e;
  if (vec && launch_round_tma<RoundKind::kAccumulate>(acc, delta, goff, n, seed, dev, stream, &e)) return e;
  if (vec) {
    const uint64_t ntiles = n / kTile;
    const unsigned blocks = ntiles ? grid_for(ntiles * kThreads, dev) : grid_for(n, dev);
    return launch_pdl(accumulate_vec_kernel, blocks, kThreads, stream, acc, delta, goff, n, seed);
  }
  return launch_pdl(accumulate_scalar_kernel, grid_for(n, dev), kThreads, stream, acc, delta, goff, n, seed);
}

cudaError_t launch_noise(uint32_t* out, uint64_t first, uint64_t n, uint32_t seed, const DeviceInfo& dev,
                         cudaStream_t stream) {
  return launch_pdl(noise_kernel, grid_for(n, dev), kThreads, stream, out, first, n, seed);
}

}  // namespace mpk
