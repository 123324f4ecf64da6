// mp_api.cu — the C ABI declared in include/mp_adamw.h: argument checks,
// host-side scalars (bias corrections, decay segments) and kernel launches.
// Nothing here synchronises, allocates device memory, prints or exits.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <vector>

#include "mp_adamw.h"
#include "mp_device.cuh"
#include "mp_internal.h"

namespace {

constexpr uint64_t kMaxN = 1ull << 62;

thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return MP_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Bias correction 1 - beta^t of step t, in double, rounded once to float.
// mp_adamw_step and the device table of replayable steps both use this.
float bias_correction(float beta, int64_t t) {
  return static_cast<float>(1.0 - std::pow(static_cast<double>(beta), static_cast<double>(t)));
}

bool beta_ok(float beta) { return beta >= 0.0f && beta < 1.0f; }

constexpr int64_t kMaxBiasLen = int64_t{1} << 26;

constexpr int32_t kMaxSumsqParts = 1 << 20;  // per-rank sums one scale call adds

constexpr double kPi = 3.141592653589793;  // the double nearest pi

}  // namespace

namespace mpk {

cudaError_t device_info(DeviceInfo* out) {
  static std::atomic<int> sms_cache[64];  // 0 = not yet queried; racing callers store the same value
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int sms = (dev >= 0 && dev < 64) ? sms_cache[dev].load(std::memory_order_relaxed) : 0;
  if (sms == 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) sms_cache[dev].store(sms, std::memory_order_relaxed);
  }
  out->device = dev;
  out->sms = sms;
  return cudaSuccess;
}

int record_cuda_error(cudaError_t e) { return cuda_fail(e); }

}  // namespace mpk

extern "C" {

int mp_abi_version(void) { return MP_ABI_VERSION; }

const char* mp_status_string(int status) {
  switch (status) {
    case MP_OK: return "MP_OK";
    case MP_ERR_NULL: return "MP_ERR_NULL: a required pointer is NULL";
    case MP_ERR_ALIGN: return "MP_ERR_ALIGN: a pointer is not aligned to its element size";
    case MP_ERR_TABLE: return "MP_ERR_TABLE: tensor table malformed or not covering the range";
    case MP_ERR_RANGE: return "MP_ERR_RANGE: a size, step or hyperparameter is out of range";
    case MP_ERR_NONFINITE: return "MP_ERR_NONFINITE: the clip scale was NaN or Inf; nothing was written";
    case MP_ERR_CUDA: return "MP_ERR_CUDA: a CUDA runtime call failed";
    case MP_ERR_WORKSPACE: return "MP_ERR_WORKSPACE: workspace missing or too small";
    case MP_SKIPPED_OUTLIER: return "MP_SKIPPED_OUTLIER: the grad-norm z-score was above the threshold; step skipped";
    case MP_ERR_ACCESS: return "MP_ERR_ACCESS: host buffer is not page-locked memory the device can read";
    default: return "unknown mp_status";
  }
}

int mp_last_cuda_error(void) { return g_last_cuda_error; }

size_t mp_grad_norm_workspace_bytes(uint64_t n) {
  mpk::DeviceInfo dev;
  if (mpk::device_info(&dev) != cudaSuccess) return 0;
  // The scalar path (unaligned grads) uses the most blocks for a given n.
  return sizeof(double) * static_cast<size_t>(mpk::norm_blocks(n, false, dev));
}

int mp_grad_norm(const uint16_t* grads, uint64_t n, float clip, void* workspace, size_t workspace_bytes,
                 float* d_norm, float* d_scale, double* d_sumsq, void* stream) {
  if ((n != 0 && grads == nullptr) || d_norm == nullptr || d_scale == nullptr) return MP_ERR_NULL;
  if (workspace == nullptr) return MP_ERR_WORKSPACE;
  if (!aligned(grads, 2) || !aligned(workspace, 8) || !aligned(d_norm, 4) || !aligned(d_scale, 4) ||
      !aligned(d_sumsq, 8))
    return MP_ERR_ALIGN;
  if (!(clip > 0.0f) || !std::isfinite(clip) || n > kMaxN) return MP_ERR_RANGE;
  mpk::DeviceInfo dev;
  cudaError_t e = mpk::device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const bool vec = aligned(grads, 16);
  const int nb = mpk::norm_blocks(n, vec, dev);
  if (workspace_bytes < sizeof(double) * static_cast<size_t>(nb)) return MP_ERR_WORKSPACE;
  e = mpk::launch_norm(grads, n, vec, static_cast<double*>(workspace), nb, clip, d_norm, d_scale, d_sumsq,
                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return MP_OK;
}

int mp_grad_sumsq(const uint16_t* grads, uint64_t n, void* workspace, size_t workspace_bytes, double* d_sumsq,
                  void* stream) {
  if ((n != 0 && grads == nullptr) || d_sumsq == nullptr) return MP_ERR_NULL;
  if (workspace == nullptr) return MP_ERR_WORKSPACE;
  if (!aligned(grads, 2) || !aligned(workspace, 8) || !aligned(d_sumsq, 8)) return MP_ERR_ALIGN;
  if (n > kMaxN) return MP_ERR_RANGE;
  mpk::DeviceInfo dev;
  cudaError_t e = mpk::device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const bool vec = aligned(grads, 16);
  const int nb = mpk::norm_blocks(n, vec, dev);
  if (workspace_bytes < sizeof(double) * static_cast<size_t>(nb)) return MP_ERR_WORKSPACE;
  e = mpk::launch_norm(grads, n, vec, static_cast<double*>(workspace), nb, 1.0f, nullptr, nullptr, d_sumsq,
                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return MP_OK;
}

int mp_clip_scale_from_sumsq(const double* d_sumsq, int32_t count, float clip, float* d_norm, float* d_scale,
                             double* d_total, void* stream) {
  if (d_sumsq == nullptr || d_norm == nullptr || d_scale == nullptr) return MP_ERR_NULL;
  if (!aligned(d_sumsq, 8) || !aligned(d_norm, 4) || !aligned(d_scale, 4) || !aligned(d_total, 8))
    return MP_ERR_ALIGN;
  if (count < 1 || count > kMaxSumsqParts || !(clip > 0.0f) || !std::isfinite(clip)) return MP_ERR_RANGE;
  const cudaError_t e = mpk::launch_scale_from_sumsq(d_sumsq, count, clip, d_norm, d_scale, d_total,
                                                     static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return MP_OK;
}

int mp_lr_at(const mp_lr_schedule_t* s, int64_t t, float* lr) {
  if (s == nullptr || lr == nullptr) return MP_ERR_NULL;
  const bool decays = s->kind != MP_LR_CONSTANT;
  if (s->kind < MP_LR_CONSTANT || s->kind > MP_LR_WSD || s->reserved != 0 || s->warmup < 0 || t < 1 ||
      (decays && s->total <= s->warmup) || !std::isfinite(s->lr_max) || !std::isfinite(s->lr_min) ||
      (s->kind == MP_LR_WSD && !(s->decay_frac > 0.0f && s->decay_frac <= 1.0f)))
    return MP_ERR_RANGE;
  const double peak = s->lr_max, floor_lr = s->lr_min;
  if (t <= s->warmup) {  // linear warm-up, reaching the peak at t = warmup
    *lr = static_cast<float>(peak * static_cast<double>(t) / static_cast<double>(s->warmup));
    return MP_OK;
  }
  if (!decays) {
    *lr = s->lr_max;
    return MP_OK;
  }
  const double span = static_cast<double>(s->total - s->warmup);
  const double p = std::fmin(1.0, static_cast<double>(t - s->warmup) / span);  // progress after warm-up
  double out = peak;
  switch (s->kind) {
    case MP_LR_COSINE:
      out = floor_lr + (peak - floor_lr) * (1.0 + std::cos(kPi * p)) / 2.0;
      break;
    case MP_LR_LINEAR:
      out = peak - (peak - floor_lr) * p;
      break;
    default: {  // MP_LR_WSD: stable, then linear over the last fraction
      const double f = s->decay_frac, start = 1.0 - f;
      out = p <= start ? peak : peak - (peak - floor_lr) * (p - start) / f;
      break;
    }
  }
  *lr = static_cast<float>(out);
  return MP_OK;
}

}  // extern "C"

namespace {

// Checks the range and the tensor table (sorted, contiguous from 0, flags in
// {0, 1}, covering [global_offset, global_offset + n)) and lists the decay
// segments over the range: maximal runs of equal flag, so flags alternate;
// seg_end[s] is one past segment s. No CUDA call.
int table_segments(uint64_t global_offset, uint64_t n, const mp_tensor_t* table, int32_t n_tensors,
                   std::vector<uint64_t>* seg_end, std::vector<int>* seg_flag) {
  if (n > kMaxN || global_offset > kMaxN - n) return MP_ERR_RANGE;
  if (table == nullptr) return MP_ERR_NULL;
  if (n_tensors < 1) return MP_ERR_TABLE;
  uint64_t off = 0;
  for (int32_t k = 0; k < n_tensors; ++k) {
    const mp_tensor_t& T = table[k];
    if (T.offset != off || T.size > kMaxN || (T.decay != 0 && T.decay != 1) || T.reserved != 0)
      return MP_ERR_TABLE;
    off += T.size;
    if (off > kMaxN) return MP_ERR_TABLE;
  }
  const uint64_t lo = global_offset, hi = global_offset + n;
  if (off < hi) return MP_ERR_TABLE;
  seg_end->clear();
  seg_flag->clear();
  for (int32_t k = 0; k < n_tensors; ++k) {
    const uint64_t a = table[k].offset, b = table[k].offset + table[k].size;
    if (b <= lo || a >= hi || a == b) continue;
    const uint64_t end = b < hi ? b : hi;
    if (!seg_flag->empty() && seg_flag->back() == table[k].decay) {
      seg_end->back() = end;
    } else {
      seg_end->push_back(end);
      seg_flag->push_back(table[k].decay);
    }
  }
  return MP_OK;
}

// One step launch: elements [c0, c1) and decay segments s0 .. last.
struct Chunk {
  uint64_t c0, c1;
  size_t s0, last;
};

// How a step over [lo, hi) with these segments is split into launches: at
// most kMaxLaunchElems elements (near-equal chunks of whole tiles) and at
// most kSegCapLarge segments each; chunk starts stay multiples of 4
// elements from lo so vector alignment is preserved.
std::vector<Chunk> split_launches(uint64_t lo, uint64_t hi, const std::vector<uint64_t>& seg_end) {
  std::vector<Chunk> out;
  const size_t ns = seg_end.size();
  if (hi <= lo || ns == 0) return out;
  const uint64_t pieces = (hi - lo + mpk::kMaxLaunchElems - 1) / mpk::kMaxLaunchElems;
  const uint64_t tile = static_cast<uint64_t>(mpk::kTile);
  const uint64_t chunk = ((hi - lo + pieces - 1) / pieces + tile - 1) / tile * tile;
  uint64_t c0 = lo;
  size_t s0 = 0;
  while (c0 < hi) {
    uint64_t c1 = hi - c0 > chunk ? c0 + chunk : hi;
    if (ns - s0 > mpk::kSegCapLarge) {
      // Cut at the start of segment s0 + CAP - 1 at the latest, rounded down
      // to a multiple of 4 from lo. Segments s0+1 .. s0+CAP-2 hold >= 1
      // element each, so the chunk keeps >= 1020 elements and at most CAP - 1
      // segments.
      const uint64_t cut = seg_end[s0 + mpk::kSegCapLarge - 2];
      const uint64_t c1s = lo + ((cut - lo) & ~static_cast<uint64_t>(3));
      if (c1s < c1) c1 = c1s;
    }
    size_t last = s0;
    while (seg_end[last] < c1) ++last;  // the segment holding element c1 - 1
    out.push_back(Chunk{c0, c1, s0, last});
    c0 = c1;
    while (s0 < ns && seg_end[s0] <= c0) ++s0;
  }
  return out;
}

// A validated step: decay segments over [lo, hi) and the launch scalars.
struct StepPlan {
  std::vector<uint64_t> seg_end;
  std::vector<int> seg_flag;
  mpk::StepArgs base{};
  uint64_t lo = 0, hi = 0;
  bool vec = false;
};

// Argument checks, host scalars and decay segments of one AdamW step. Makes
// no CUDA call, so a failure leaves the stream untouched.
int plan_step(uint16_t* params, const uint16_t* grads, float* master, float* m, float* v, uint64_t global_offset,
              uint64_t n, const mp_tensor_t* table, int32_t n_tensors, float lr, float beta1, float beta2, float eps,
              float weight_decay, const float* d_grad_scale, int32_t t, uint32_t seed, int32_t* d_status,
              StepPlan* plan) {
  if (params == nullptr || grads == nullptr || m == nullptr || v == nullptr || table == nullptr)
    return MP_ERR_NULL;
  if (!aligned(params, 2) || !aligned(grads, 2) || !aligned(master, 4) || !aligned(m, 4) || !aligned(v, 4) ||
      !aligned(d_grad_scale, 4) || !aligned(d_status, 4))
    return MP_ERR_ALIGN;
  if (!std::isfinite(lr) || !std::isfinite(eps) || !std::isfinite(weight_decay) || !(beta1 >= 0.0f) ||
      !(beta1 < 1.0f) || !(beta2 >= 0.0f) || !(beta2 < 1.0f) || t < 1)
    return MP_ERR_RANGE;
  const int st = table_segments(global_offset, n, table, n_tensors, &plan->seg_end, &plan->seg_flag);
  if (st != MP_OK) return st;
  plan->lo = global_offset;
  plan->hi = global_offset + n;

  mpk::StepArgs& base = plan->base;
  base.d_scale = d_grad_scale;
  base.d_status = d_status;
  base.lr = lr;
  base.beta1 = beta1;
  base.beta2 = beta2;
  base.eps = eps;
  base.wd = weight_decay;
  base.bc1 = bias_correction(beta1, t);
  base.bc2 = bias_correction(beta2, t);
  base.seed = seed;
  plan->vec = aligned(params, 8) && aligned(grads, 8) && aligned(master, 16) && aligned(m, 16) && aligned(v, 16);
  return MP_OK;
}

// One launch per chunk of split_launches.
cudaError_t launch_step(const StepPlan& plan, uint16_t* params, const uint16_t* grads, float* master, float* m,
                        float* v, const mpk::DeviceInfo& dev, cudaStream_t s) {
  const std::vector<uint64_t>& seg_end = plan.seg_end;
  for (const Chunk& c : split_launches(plan.lo, plan.hi, seg_end)) {
    mpk::StepArgs a = plan.base;
    const uint64_t d = c.c0 - plan.lo;
    a.params = params + d;
    a.grads = grads + d;
    a.master = master ? master + d : nullptr;
    a.m = m + d;
    a.v = v + d;
    a.n = c.c1 - c.c0;
    a.goff = c.c0;
    a.nseg = static_cast<uint32_t>(c.last - c.s0 + 1);
    a.first_decay = static_cast<uint32_t>(plan.seg_flag[c.s0]);
    std::vector<uint64_t> ends(seg_end.begin() + c.s0, seg_end.begin() + c.last + 1);
    ends.back() = c.c1;
    const cudaError_t e = mpk::launch_adamw(a, ends.data(), plan.vec, dev, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

extern "C" {

int mp_adamw_step(uint16_t* params, const uint16_t* grads, float* master, float* m, float* v,
                  uint64_t global_offset, uint64_t n, const mp_tensor_t* table, int32_t n_tensors,
                  float lr, float beta1, float beta2, float eps, float weight_decay, const float* d_grad_scale,
                  int32_t t, uint32_t seed, int32_t* d_status, void* stream) {
  if (n == 0) return MP_OK;
  StepPlan plan;
  const int st = plan_step(params, grads, master, m, v, global_offset, n, table, n_tensors, lr, beta1, beta2, eps,
                           weight_decay, d_grad_scale, t, seed, d_status, &plan);
  if (st != MP_OK) return st;
  mpk::DeviceInfo dev;
  cudaError_t e = mpk::device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  e = launch_step(plan, params, grads, master, m, v, dev, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return MP_OK;
}

}  // extern "C"

namespace {

// mp_optimizer_step and mp_optimizer_step_graph: with `clock`, the norm's
// finalize kernel advances the device step counter and the update reads lr,
// seed and bias corrections from the device state (t, seed and hyper->lr are
// then unused).
int optimizer_step(uint16_t* params, uint16_t* grads, const uint16_t* host_grads, float* master, float* m,
                   float* v, uint64_t n, const mp_tensor_t* table, int32_t n_tensors, const mp_hyper_t* hyper,
                   int32_t t, uint32_t seed, const mpk::StepClock* clock, void* workspace, size_t workspace_bytes,
                   void* outlier_state, float outlier_z, double* d_z, float* d_norm, float* d_scale,
                   int32_t* d_status, float* host_norm, void* stream) {
  if (hyper == nullptr || d_norm == nullptr || d_scale == nullptr) return MP_ERR_NULL;
  if (workspace == nullptr) return MP_ERR_WORKSPACE;
  if (!aligned(workspace, 8) || !aligned(d_norm, 4) || !aligned(d_scale, 4) || !aligned(outlier_state, 8) ||
      !aligned(d_z, 8) || !aligned(host_grads, 2) || !aligned(host_norm, 4))
    return MP_ERR_ALIGN;
  if (!(hyper->clip > 0.0f) || !std::isfinite(hyper->clip)) return MP_ERR_RANGE;
  StepPlan plan;
  if (n != 0) {
    const float lr = clock != nullptr ? 0.0f : hyper->lr;
    const int st = plan_step(params, grads, master, m, v, 0, n, table, n_tensors, lr, hyper->beta1,
                             hyper->beta2, hyper->eps, hyper->weight_decay, d_scale, t, seed, d_status, &plan);
    if (st != MP_OK) return st;
    if (clock != nullptr) plan.base.dstate = clock->state;
  }
  // Host gradients must be page-locked: their device-visible address is read
  // by the norm kernel, which also writes the device copy into `grads`.
  const uint16_t* src = grads;
  if (host_grads != nullptr && n != 0) {
    cudaPointerAttributes attr{};
    const cudaError_t e = cudaPointerGetAttributes(&attr, host_grads);
    if (e != cudaSuccess) {
      cudaGetLastError();  // clear the non-sticky error this query may leave
      return MP_ERR_ACCESS;
    }
    if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) return MP_ERR_ACCESS;
    src = static_cast<const uint16_t*>(attr.devicePointer);
  }
  mpk::DeviceInfo dev;
  cudaError_t e = mpk::device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const bool copy = host_grads != nullptr && n != 0;
  const bool vec = aligned(src, 16) && (!copy || aligned(grads, 16));
  const int nb = mpk::norm_blocks(n, vec, dev);
  if (workspace_bytes < sizeof(double) * static_cast<size_t>(nb)) return MP_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The cluster kernel reads the update's gradients where the norm reads
  // them (src), with 8-B vector loads like the update kernel's.
  const bool small = n != 0 && n <= mpk::kSmallMaxN && plan.vec && aligned(src, 8) &&
                     plan.seg_end.size() <= mpk::kSegCapSmall && nb <= mpk::kSmallClusterCtas &&
                     mpk::small_step_available(dev, master != nullptr);
  if (small) {  // one cluster launch, the same results as the three launches below
    mpk::StepArgs a = plan.base;
    a.params = params;
    a.grads = grads;
    a.master = master;
    a.m = m;
    a.v = v;
    a.n = n;
    a.goff = 0;
    a.nseg = static_cast<uint32_t>(plan.seg_end.size());
    a.first_decay = static_cast<uint32_t>(plan.seg_flag[0]);
    const mpk::SmallArgs sa{src, copy ? grads : nullptr, nb, vec ? 1 : 0, hyper->clip, d_norm, d_scale,
                            clock != nullptr ? *clock : mpk::StepClock{nullptr, nullptr, 0, nullptr},
                            outlier_state, outlier_z, d_z};
    e = mpk::launch_small_step(a, sa, plan.seg_end.data(), s);
  } else {
    e = mpk::launch_norm(src, n, vec, static_cast<double*>(workspace), nb, hyper->clip, d_norm, d_scale,
                         nullptr, s, copy ? grads : nullptr, clock);
    if (e == cudaSuccess && outlier_state != nullptr)
      e = mpk::launch_outlier_check(outlier_state, d_norm, outlier_z, d_scale, d_z, d_status, s);
    if (e == cudaSuccess && n != 0) e = launch_step(plan, params, grads, master, m, v, dev, s);
  }
  if (e == cudaSuccess && host_norm != nullptr)
    e = cudaMemcpyAsync(host_norm, d_norm, sizeof(float), cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return MP_OK;
}

}  // namespace

extern "C" {

int mp_optimizer_step(uint16_t* params, uint16_t* grads, const uint16_t* host_grads, float* master, float* m,
                      float* v, uint64_t n, const mp_tensor_t* table, int32_t n_tensors, const mp_hyper_t* hyper,
                      int32_t t, uint32_t seed, void* workspace, size_t workspace_bytes, void* outlier_state,
                      float outlier_z, double* d_z, float* d_norm, float* d_scale, int32_t* d_status,
                      float* host_norm, void* stream) {
  return optimizer_step(params, grads, host_grads, master, m, v, n, table, n_tensors, hyper, t, seed, nullptr,
                        workspace, workspace_bytes, outlier_state, outlier_z, d_z, d_norm, d_scale, d_status,
                        host_norm, stream);
}

int64_t mp_bias_table_len(float beta1, float beta2) {
  if (!beta_ok(beta1) || !beta_ok(beta2)) return 0;
  for (int64_t t = 1; t <= kMaxBiasLen; ++t)
    if (bias_correction(beta1, t) == 1.0f && bias_correction(beta2, t) == 1.0f) return t;
  return 0;
}

int mp_bias_table(float beta1, float beta2, int64_t len, float* out) {
  if (out == nullptr) return MP_ERR_NULL;
  if (!beta_ok(beta1) || !beta_ok(beta2) || len < 1 || len > kMaxBiasLen) return MP_ERR_RANGE;
  for (int64_t t = 1; t <= len; ++t) {
    out[2 * (t - 1)] = bias_correction(beta1, t);
    out[2 * (t - 1) + 1] = bias_correction(beta2, t);
  }
  return MP_OK;
}

int mp_optimizer_step_graph(uint16_t* params, uint16_t* grads, const uint16_t* host_grads, float* master,
                            float* m, float* v, uint64_t n, const mp_tensor_t* table, int32_t n_tensors,
                            const mp_hyper_t* hyper, mp_step_state_t* d_state, const float* d_bias,
                            int64_t bias_len, void* workspace, size_t workspace_bytes, void* outlier_state,
                            float outlier_z, double* d_z, float* d_norm, float* d_scale, int32_t* d_status,
                            float* host_norm, void* stream) {
  if (d_state == nullptr || d_bias == nullptr) return MP_ERR_NULL;
  if (!aligned(d_state, 16) || !aligned(d_bias, 4)) return MP_ERR_ALIGN;
  if (bias_len < 1 || bias_len > kMaxBiasLen) return MP_ERR_RANGE;
  const mpk::StepClock clock{d_state, d_bias, bias_len, d_status};
  return optimizer_step(params, grads, host_grads, master, m, v, n, table, n_tensors, hyper, 1, 0, &clock,
                        workspace, workspace_bytes, outlier_state, outlier_z, d_z, d_norm, d_scale, d_status,
                        host_norm, stream);
}

int mp_step_launches(uint64_t global_offset, uint64_t n, const mp_tensor_t* table, int32_t n_tensors,
                     mp_launch_t* out, int64_t capacity, int64_t* count) {
  if (count == nullptr || (capacity > 0 && out == nullptr)) return MP_ERR_NULL;
  if (capacity < 0) return MP_ERR_RANGE;
  std::vector<uint64_t> seg_end;
  std::vector<int> seg_flag;
  const int st = table_segments(global_offset, n, table, n_tensors, &seg_end, &seg_flag);
  if (st != MP_OK) return st;
  const std::vector<Chunk> chunks = split_launches(global_offset, global_offset + n, seg_end);
  *count = static_cast<int64_t>(chunks.size());
  for (size_t i = 0; i < chunks.size() && static_cast<int64_t>(i) < capacity; ++i) {
    out[i].offset = chunks[i].c0;
    out[i].size = chunks[i].c1 - chunks[i].c0;
    out[i].segments = static_cast<uint32_t>(chunks[i].last - chunks[i].s0 + 1);
    out[i].first_decay = static_cast<uint32_t>(seg_flag[chunks[i].s0]);
  }
  return MP_OK;
}

int mp_stochastic_round(uint16_t* out, const float* in, uint64_t global_offset, uint64_t n, uint32_t seed,
                        void* stream) {
  if (n == 0) return MP_OK;
  if (out == nullptr || in == nullptr) return MP_ERR_NULL;
  if (!aligned(out, 2) || !aligned(in, 4)) return MP_ERR_ALIGN;
  if (n > kMaxN || global_offset > kMaxN - n) return MP_ERR_RANGE;
  mpk::DeviceInfo dev;
  cudaError_t e = mpk::device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const bool vec = aligned(in, 16) && aligned(out, 8);
  e = mpk::launch_sr(out, in, global_offset, n, seed, vec, dev, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return MP_OK;
}

int mp_stochastic_round_fp16(uint16_t* out, const float* in, uint64_t global_offset, uint64_t n, uint32_t seed,
                             void* stream) {
  if (n == 0) return MP_OK;
  if (out == nullptr || in == nullptr) return MP_ERR_NULL;
  if (!aligned(out, 2) || !aligned(in, 4)) return MP_ERR_ALIGN;
  if (n > kMaxN || global_offset > kMaxN - n) return MP_ERR_RANGE;
  mpk::DeviceInfo dev;
  cudaError_t e = mpk::device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const bool vec = aligned(in, 16) && aligned(out, 8);
  e = mpk::launch_sr_fp16(out, in, global_offset, n, seed, vec, dev, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return MP_OK;
}

int mp_accumulate_sr(uint16_t* acc, const float* delta, uint64_t global_offset, uint64_t n, uint32_t seed,
                     void* stream) {
  if (n == 0) return MP_OK;
  if (acc == nullptr || delta == nullptr) return MP_ERR_NULL;
  if (!aligned(acc, 2) || !aligned(delta, 4)) return MP_ERR_ALIGN;
  if (n > kMaxN || global_offset > kMaxN - n) return MP_ERR_RANGE;
  mpk::DeviceInfo dev;
  cudaError_t e = mpk::device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const bool vec = aligned(delta, 16) && aligned(acc, 8);
  e = mpk::launch_accumulate_sr(acc, delta, global_offset, n, seed, vec, dev, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return MP_OK;
}

int mp_noise_u32(uint32_t* out, uint64_t first_index, uint64_t n, uint32_t seed, void* stream) {
  if (n == 0) return MP_OK;
  if (out == nullptr) return MP_ERR_NULL;
  if (!aligned(out, 4)) return MP_ERR_ALIGN;
  if (n > kMaxN) return MP_ERR_RANGE;
  mpk::DeviceInfo dev;
  cudaError_t e = mpk::device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  e = mpk::launch_noise(out, first_index, n, seed, dev, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return MP_OK;
}

}  // extern "C"
