/*
 * mp_adamw.h — C ABI of libmpadamw.so: the mixed-precision optimizer step of
 * bf16 LLM training on one GB300 (sm_103a).
 *
 * Sources (web pages; cited by title and section):
 *   [LLMC]  llm.c code walk-through, ch. 04 "Multi-GPU and mixed precision"
 *           (ai-reference-codex.pages.dev): §2.1 precision table, §2.2 AdamW
 *           kernel, §2.3 stochastic rounding, §3.2 ZeRO-1 shards, §4 train step.
 *   [CMU13] CMU 11-667 lecture 13 notes, "Scaling up LLMs: optimization and
 *           parallel training" (semidirectx.com): §1.6-1.7 Adam/AdamW details,
 *           §2.3 fp32 master weights, §7.3 exercises 1 and 5.
 *   [DIST3] "LLM distributed training: CUDA/ROCm multi-GPU, part 3": §3.1
 *           ZeRO stage 1 (the shard is a contiguous index range).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - bf16 values travel as their raw 16-bit patterns (uint16_t).
 *  - Every pointer is a DEVICE pointer unless marked "host". The caller owns
 *    every buffer and the stream; the library keeps no pointer after return.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Every call only enqueues work on `stream` and returns; nothing here
 *    synchronises the device or the stream.
 *  - Calls validate their arguments on the host before any launch. On an
 *    error they return a status != MP_OK and enqueue nothing: no output
 *    buffer is touched.
 *  - Element counts and offsets are 64-bit: a parameter set may exceed 2^32
 *    elements. A "global index" is an element's position in the whole flat
 *    parameter buffer; a call may cover only the range
 *    [global_offset, global_offset + n) of it (a ZeRO-1 shard, [LLMC] §3.2,
 *    [DIST3] §3.1), and every pointer then addresses element global_offset.
 *  - Pointers must be aligned to their element size (2 B for bf16, 4 B for
 *    fp32, 8 B for fp64) or the call returns MP_ERR_ALIGN. Buffers that are
 *    also 16-B aligned take the vectorised kernels; others take scalar
 *    kernels that compute bit-identical updates and roundings more slowly
 *    (the gradient norm's two paths differ in rounding: see mp_grad_norm).
 *  - Input and output buffers of one call must not overlap (params, grads,
 *    master, m and v are distinct arrays), and every device pointer must
 *    belong to the current device (cudaSetDevice) of the calling thread.
 *  - Nothing in the library calls exit(), prints, or allocates device memory.
 */
#ifndef MP_ADAMW_H
#define MP_ADAMW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MP_ABI_VERSION 1

/* One tensor of the flat parameter buffer. Offsets and sizes are global
 * element indices. `decay` is 1 for tensors that take weight decay and 0 for
 * those that do not; [LLMC] §2.2 decays embeddings and matrices (2D tensors)
 * and exempts LayerNorm weights and biases (1D tensors). */
typedef struct mp_tensor {
    uint64_t offset;
    uint64_t size;
    int32_t decay;
    int32_t reserved; /* must be 0 */
} mp_tensor_t;

typedef enum mp_status {
    MP_OK = 0,
    MP_ERR_NULL = 1,      /* a required pointer is NULL                          */
    MP_ERR_ALIGN = 2,     /* a pointer is not aligned to its element size        */
    MP_ERR_TABLE = 3,     /* tensor table malformed or not covering the range   */
    MP_ERR_RANGE = 4,     /* a size, step or hyperparameter is out of range      */
    MP_ERR_NONFINITE = 5, /* device-reported: the clip scale was NaN or Inf      */
    MP_ERR_CUDA = 6,      /* a CUDA runtime call failed (see mp_last_cuda_error) */
    MP_ERR_WORKSPACE = 7, /* workspace missing or smaller than required          */
    MP_SKIPPED_OUTLIER = 8, /* device-reported: the outlier check skipped the step */
    MP_ERR_ACCESS = 9     /* a host buffer is not page-locked memory the device can read */
} mp_status_t;

/* Optimizer hyperparameters of mp_optimizer_step. */
typedef struct mp_hyper {
    float lr, beta1, beta2, eps, weight_decay;
    float clip; /* clip threshold of the grad norm (the train step uses 1.0) */
} mp_hyper_t;

/* ABI version this library was built with (MP_ABI_VERSION). */
int mp_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* mp_status_string(int status);

/* The cudaError_t of the last failing CUDA call made by the calling host
 * thread inside this library, 0 if none. Thread-local. */
int mp_last_cuda_error(void);

/* ---------------------------------------------------------------------------
 * Gradient norm and clip scale — [LLMC] §4 ("grad_norm = global norm";
 * "grad_scale = min(1, 1.0/grad_norm)", i.e. clipping to norm 1.0).
 *
 *   sumsq = sum over all i < n of (float)grads[i]^2    (all tensors, 1D too)
 *   norm  = (float) sqrt(sumsq)
 *   scale = NaN                        if norm is NaN or Inf
 *         = min(1, clip / norm)        otherwise (fp32 divide; norm 0 -> 1)
 *
 * The kernel squares in fp32 (exact for |g| in [2^-63, 2^64)), sums each
 * thread's terms with compensation, and reduces across threads and blocks in
 * fp64 in a fixed order; a block whose fp32 partial is non-finite or below
 * 2^-60 recomputes its share in fp64. Gradients that are 16-B aligned are
 * read as 8-element vectors whose squares are added pairwise in fp32;
 * others element by element, so the two differ in rounding. The result is
 * bit-identical on every run with the same n and the same alignment class
 * on the same GPU model; its relative error against an fp64 sum is below
 * 1e-6 for any finite input.
 *
 *   grads       bf16[n], device, read only.
 *   n           element count; 0 gives sumsq 0, norm 0, scale 1.
 *   clip        clip threshold, finite and > 0 (the train step uses 1.0).
 *   workspace   device scratch of at least mp_grad_norm_workspace_bytes(n)
 *               bytes, 8-B aligned; overwritten, no initial contents needed;
 *               must not be shared with another call in flight.
 *   d_norm      float[1], device, written.
 *   d_scale     float[1], device, written (feeds mp_adamw_step).
 *   d_sumsq     double[1], device, written; may be NULL.
 * Launches: 16-B aligned gradients of at least 16,384 elements per SM have
 * each first-level block read one contiguous run of them, staged through
 * shared memory by the TMA engine (49 KB per block); it adds the same squares
 * in the same order as the register kernel that reads host gradients
 * (mp_optimizer_step's host_grads), so the result is the same bits. If one of
 * its bounded waits gives up (only a fault of the GPU or of the library can
 * cause that), the norm and the scale come out NaN.
 * Errors: MP_ERR_NULL, MP_ERR_ALIGN, MP_ERR_RANGE (clip), MP_ERR_WORKSPACE,
 *         MP_ERR_CUDA.
 * ------------------------------------------------------------------------- */
size_t mp_grad_norm_workspace_bytes(uint64_t n);

int mp_grad_norm(const uint16_t* grads, uint64_t n, float clip,
                 void* workspace, size_t workspace_bytes,
                 float* d_norm, float* d_scale, double* d_sumsq,
                 void* stream);

/* ---------------------------------------------------------------------------
 * The norm in two halves, for ZeRO-1 — [LLMC] §4: under ZeRO-1 each rank
 * takes the sum of squares of its own gradient shard only (after the
 * reduce-scatter of §3.2), and the per-rank sums are combined across ranks
 * before the clip scale is taken; [CMU13] §5.2: ZeRO-1 computes what data
 * parallelism computes.
 *
 * mp_grad_sumsq: sumsq of grads[0, n) exactly as mp_grad_norm computes it
 * (the same kernels, the same bits), written to *d_sumsq; no norm or scale.
 *   grads, n, workspace, workspace_bytes, stream   as mp_grad_norm.
 *   d_sumsq   double[1], device, written.
 * Errors: MP_ERR_NULL, MP_ERR_ALIGN, MP_ERR_RANGE, MP_ERR_WORKSPACE,
 *         MP_ERR_CUDA.
 *
 * mp_clip_scale_from_sumsq: combines `count` sums of squares (one per rank,
 * gathered by the caller's collective into d_sumsq[0..count) in rank order):
 *   S     = d_sumsq[0] + d_sumsq[1] + ... + d_sumsq[count-1]
 *           (fp64, left to right: every rank that passes the same values gets
 *           the same bits, whatever its own rank)
 *   norm  = (float) sqrt(S);   scale = as mp_grad_norm (NaN if norm is not
 *           finite, else min(1, clip / norm))
 * With count == 1 and mp_grad_sumsq's output this is mp_grad_norm's result.
 *   d_sumsq   double[count], device, read only.
 *   count     1 .. 2^20.
 *   clip      finite and > 0.
 *   d_norm, d_scale   float[1], device, written.
 *   d_total   double[1], device, written (S); may be NULL.
 * One single-thread kernel; nothing is allocated.
 * Errors: MP_ERR_NULL, MP_ERR_ALIGN, MP_ERR_RANGE, MP_ERR_CUDA.
 * ------------------------------------------------------------------------- */
int mp_grad_sumsq(const uint16_t* grads, uint64_t n, void* workspace, size_t workspace_bytes,
                  double* d_sumsq, void* stream);

int mp_clip_scale_from_sumsq(const double* d_sumsq, int32_t count, float clip,
                             float* d_norm, float* d_scale, double* d_total, void* stream);

/* ---------------------------------------------------------------------------
 * Learning-rate schedules — [LLMC] §4 names four (cosine, linear, constant,
 * WSD) and prints no formula. The learning rate of the 1-based step t (the t
 * mp_adamw_step takes), computed on the host in double and rounded to float
 * once:
 *   t <= warmup:  lr_max * t / warmup                      (linear warm-up)
 *   afterwards, p = min(1, (t - warmup) / (total - warmup)):
 *     MP_LR_CONSTANT  lr_max
 *     MP_LR_COSINE    lr_min + (lr_max - lr_min) * (1 + cos(pi * p)) / 2
 *     MP_LR_LINEAR    lr_max - (lr_max - lr_min) * p
 *     MP_LR_WSD       lr_max while p <= 1 - decay_frac (warm-up, stable),
 *                     then lr_max - (lr_max - lr_min) * (p - (1 - decay_frac))
 *                     / decay_frac: linear to lr_min over the last fraction
 * Steps past `total` keep the last value. Host only; no CUDA call.
 *   s    host struct: kind, warmup >= 0, total > warmup (not used by
 *        MP_LR_CONSTANT), finite lr_max and lr_min, decay_frac in (0, 1]
 *        (MP_LR_WSD only), reserved fields 0.
 *   t    >= 1.
 *   lr   host float[1], written.
 * Errors: MP_ERR_NULL, MP_ERR_RANGE (invalid schedule or t < 1).
 * ------------------------------------------------------------------------- */
typedef enum mp_lr_kind {
    MP_LR_CONSTANT = 0,
    MP_LR_COSINE = 1,
    MP_LR_LINEAR = 2,
    MP_LR_WSD = 3
} mp_lr_kind_t;

typedef struct mp_lr_schedule {
    int32_t kind;      /* mp_lr_kind_t */
    int32_t reserved;  /* must be 0 */
    int64_t warmup;    /* warm-up steps */
    int64_t total;     /* steps of the run */
    float lr_max, lr_min;
    float decay_frac;  /* MP_LR_WSD: fraction of the post-warm-up steps that decays */
    float reserved2;   /* must be 0 (not checked) */
} mp_lr_schedule_t;

int mp_lr_at(const mp_lr_schedule_t* s, int64_t t, float* lr);

/* ---------------------------------------------------------------------------
 * AdamW step with stochastic-rounding write-back — [LLMC] §2.2 (update),
 * §2.3 (rounding), §4 (t = step + 1); [CMU13] §1.7 (bias correction,
 * decoupled decay).
 *
 * Host side: bc1 = (float)(1 - beta1^t), bc2 = (float)(1 - beta2^t), both
 * computed in double and rounded once. Per element i in the range, in fp32
 * with round-to-nearest-even, no FMA contraction except the two lerps, and
 * no flush of subnormals:
 *
 *   g    = scale * (float)grads[i]
 *   m    = fma(beta1, m, fma(-beta1, g, g))           lerp(g, m, beta1)
 *   v    = fma(beta2, v, fma(-beta2, g*g, g*g))       lerp(g*g, v, beta2)
 *   mh   = m / bc1;   vh = v / bc2
 *   old  = master ? master[i] : (float)params[i]
 *   wd_e = (tensor of i).decay ? weight_decay : 0
 *   p    = old - lr * ( mh / (sqrt(vh) + eps) + wd_e * old )
 *   master[i] = p                                      (if master != NULL)
 *   params[i] = SR(p, global index of i, seed)
 *
 * SR(x, k, seed): x NaN -> 0x7FC0; otherwise b = bits(x),
 *   params = (b >> 16) + ((b & 0xFFFF) > (noise(k, seed) & 0xFFFF) ? 1 : 0)
 * i.e. the bf16 neighbour away from zero with probability (b & 0xFFFF)/65536,
 * and noise() is the counter hash documented at mp_noise_u32.
 *
 *   params      bf16[n], device, read (no-master variant) and written.
 *   grads       bf16[n], device, read only.
 *   master      fp32[n], device, read and written; NULL selects the
 *               no-master variant, which reads the old weight from params.
 *   m, v        fp32[n], device, read and written.
 *   global_offset, n   the covered global range; n == 0 is a no-op.
 *   table, n_tensors   HOST array describing the whole flat buffer: sorted,
 *               contiguous from offset 0, decay in {0,1}, reserved == 0, and
 *               covering [global_offset, global_offset + n).
 *   lr, beta1, beta2, eps, weight_decay   finite; beta1, beta2 in [0, 1).
 *   d_grad_scale  float[1], device (normally mp_grad_norm's d_scale); NULL
 *               means scale 1. If it holds NaN or Inf the kernel writes no
 *               buffer at all and stores MP_ERR_NONFINITE into *d_status
 *               unless *d_status already holds an error (the first wins).
 *   t           1-based step count (t >= 1).
 *   seed        per-step rounding seed.
 *   d_status    int32[1], device, may be NULL; written only on that device-
 *               side error, and only while it holds 0 (the caller zeroes it
 *               and reads it after a sync). MP_ERR_CUDA there means a kernel
 *               gave up waiting (one second) for its own staged copies, which
 *               only a fault of the GPU or of the library can cause.
 * Launches: ranges of at least two tiles per SM (tiles of 2,304 elements with
 * master, 3,328 without) whose arrays are 16-B aligned where the tiles start
 * run a kernel that stages whole tiles through shared memory with the TMA
 * engine (one block per SM, 129 KB or 200 KB of shared memory); others run a
 * register-only kernel. Both give the same bits.
 * Errors: MP_ERR_NULL, MP_ERR_ALIGN, MP_ERR_TABLE, MP_ERR_RANGE, MP_ERR_CUDA.
 * ------------------------------------------------------------------------- */
int mp_adamw_step(uint16_t* params, const uint16_t* grads, float* master,
                  float* m, float* v,
                  uint64_t global_offset, uint64_t n,
                  const mp_tensor_t* table, int32_t n_tensors,
                  float lr, float beta1, float beta2, float eps,
                  float weight_decay, const float* d_grad_scale,
                  int32_t t, uint32_t seed, int32_t* d_status,
                  void* stream);

/* ---------------------------------------------------------------------------
 * How mp_adamw_step splits a range into kernel launches (host only; no CUDA
 * call). Each launch covers at most 201,326,592 elements (long ranges are
 * cut into near-equal launches of whole 2048-element tiles: on GB300 one
 * persistent launch over billions of elements streams about 1 % slower) and
 * at most 1024 decay segments (the table a launch carries in its kernel
 * parameters); launch offsets stay multiples of 4 elements from
 * global_offset. The whole-step calls use the same split for their update,
 * except that a small set (n <= 32,768) runs in one cluster launch.
 *
 *   global_offset, n, table, n_tensors   as mp_adamw_step.
 *   out        host array of `capacity` entries, or NULL with capacity 0;
 *              receives the first min(capacity, count) launches in order.
 *   count      host int64[1]: the number of launches.
 * Errors: MP_ERR_NULL, MP_ERR_RANGE, MP_ERR_TABLE.
 * ------------------------------------------------------------------------- */
typedef struct mp_launch {
    uint64_t offset;      /* global index of the launch's first element */
    uint64_t size;        /* elements in the launch */
    uint32_t segments;    /* decay segments it carries */
    uint32_t first_decay; /* decay flag of its first segment (flags alternate) */
} mp_launch_t;

int mp_step_launches(uint64_t global_offset, uint64_t n, const mp_tensor_t* table, int32_t n_tensors,
                     mp_launch_t* out, int64_t capacity, int64_t* count);

/* ---------------------------------------------------------------------------
 * Stochastic rounding fp32 -> bf16 of a range — [LLMC] §2.3 (the rounding
 * rule) and §5.2 (rebuilding bf16 weights from the fp32 master with the
 * saved rounding randomness).
 *
 *   out[i] = SR(in[i], global_offset + i, seed)  for i < n   (rule above)
 *
 *   out   bf16[n], device, written.   in   fp32[n], device, read only.
 * Launches: with both arrays 16-B aligned and n at least 128 tiles of 6,144
 * elements per SM, a kernel that stages whole tiles through shared memory
 * with the TMA engine (one block per SM, 221 KB of shared memory); otherwise
 * a register-only kernel. Both give the same bits.
 * Errors: MP_ERR_NULL, MP_ERR_ALIGN, MP_ERR_RANGE, MP_ERR_CUDA.
 * ------------------------------------------------------------------------- */
int mp_stochastic_round(uint16_t* out, const float* in,
                        uint64_t global_offset, uint64_t n, uint32_t seed,
                        void* stream);

/* ---------------------------------------------------------------------------
 * Stochastic rounding fp32 -> fp16 of a range. [LLMC] §6 notes that fp16
 * stochastic rounding is unfinished upstream; this is [LLMC] §2.3's rule on
 * fp16's grid, with the same draws as the bf16 rounding:
 *
 *   out[i] = x's fp16 neighbour toward zero, or the next fp16 away from zero
 *            when floor(f * 65536) > (noise(global_offset + i, seed) & 0xFFFF),
 *            f = the discarded fraction of one fp16 step (13 exact bits for
 *            fp16 normal values; cut to 16 bits below 2^-14)
 *   |x| >= 65536 -> +-Inf (the step after the largest finite fp16 is Inf);
 *   NaN -> 0x7E00; the sign is kept.
 *
 *   out   fp16[n] patterns (uint16), device, written.   in   fp32[n], device.
 * Errors: MP_ERR_NULL, MP_ERR_ALIGN, MP_ERR_RANGE, MP_ERR_CUDA.
 * ------------------------------------------------------------------------- */
int mp_stochastic_round_fp16(uint16_t* out, const float* in,
                             uint64_t global_offset, uint64_t n, uint32_t seed,
                             void* stream);

/* ---------------------------------------------------------------------------
 * Accumulation into bf16 with stochastic rounding — [LLMC] §2.3: the same
 * rounding also writes the encoder's embedding gradients in the backward
 * pass (dwte, dwpe): the stored bf16 value is widened to fp32, the fp32
 * contribution added (one round-to-nearest addition) and the sum written
 * back by stochastic rounding, so contributions far below a bf16 step are
 * kept in expectation.
 *
 *   acc[i] = SR((float)acc[i] + delta[i], global_offset + i, seed)  for i < n
 *
 *   acc     bf16[n], device, read and written in place.
 *   delta   fp32[n], device, read only; must not overlap acc.
 * Launches: with both arrays 16-B aligned and n at least 80 tiles of 4,096
 * elements per SM, a kernel that stages whole tiles through shared memory
 * with the TMA engine (one block per SM, 147 KB of shared memory); otherwise
 * a register-only kernel. Both give the same bits.
 * Errors: MP_ERR_NULL, MP_ERR_ALIGN, MP_ERR_RANGE, MP_ERR_CUDA.
 * ------------------------------------------------------------------------- */
int mp_accumulate_sr(uint16_t* acc, const float* delta,
                     uint64_t global_offset, uint64_t n, uint32_t seed,
                     void* stream);

/* ---------------------------------------------------------------------------
 * The rounding randomness itself — [LLMC] §2.3 and §7 name SquirrelNoise5 /
 * Get2dNoiseUint. noise(k, seed) is the 2D form of SquirrelNoise5 (Squirrel
 * Eiserloh's published counter-based noise hash) at x = low 32 bits of k,
 * y = high 32 bits of k:
 *   pos = x + 198491317 * y (mod 2^32)
 *   h = pos * 0xD2A80A3F;  h += seed;      h ^= h >> 9;
 *   h += 0xA884F197;       h ^= h >> 11;
 *   h *= 0x6C736F4B;       h ^= h >> 13;
 *   h += 0xB79F3ABB;       h ^= h >> 15;
 *   h *= 0x1B56C4F5;       h ^= h >> 17;      (all mod 2^32)
 * It is keyed on the global element index, not on the launch geometry, so a
 * result does not depend on grid shape or on how the buffer is sharded.
 *
 *   out[i] = noise(first_index + i, seed)   for i < n;  out uint32[n], device.
 * Errors: MP_ERR_NULL, MP_ERR_ALIGN, MP_ERR_RANGE, MP_ERR_CUDA.
 * ------------------------------------------------------------------------- */
int mp_noise_u32(uint32_t* out, uint64_t first_index, uint64_t n,
                 uint32_t seed, void* stream);

/* ---------------------------------------------------------------------------
 * Grad-norm outlier check — [LLMC] §4: the train step keeps a window of 128
 * past grad norms and skips the update when the new norm's z-score is above
 * a threshold. This runs on the device between mp_grad_norm and
 * mp_adamw_step (one single-thread kernel, no host round trip):
 *
 *   z = (norm - mean(W)) / std(W)   W = the 128 most recent finite norms,
 *                                   population std, fp64, sums in slot order
 *   z = NaN while fewer than 128 finite norms have been seen
 *   if z_threshold > 0 and z > z_threshold:
 *       *d_scale = NaN                 (so mp_adamw_step writes nothing)
 *       *d_status = MP_SKIPPED_OUTLIER (if it was 0: the first error wins)
 *   then a finite norm joins W, replacing the oldest; a non-finite one does not.
 *
 *   d_state     device buffer of mp_outlier_state_bytes() bytes, 8-B aligned,
 *               zeroed once by mp_outlier_reset (or by the caller) before the
 *               first check; owned by the caller; one per training run.
 *   d_norm      float[1], device, read (mp_grad_norm's d_norm).
 *   z_threshold <= 0 or NaN: never skip (z is still computed).
 *   d_scale     float[1], device, read and possibly set to NaN.
 *   d_z         double[1], device, written; may be NULL.
 *   d_status    int32[1], device, may be NULL.
 * Errors: MP_ERR_NULL, MP_ERR_ALIGN, MP_ERR_CUDA.
 * ------------------------------------------------------------------------- */
size_t mp_outlier_state_bytes(void);

int mp_outlier_reset(void* d_state, void* stream);

int mp_outlier_check(void* d_state, const float* d_norm, float z_threshold,
                     float* d_scale, double* d_z, int32_t* d_status,
                     void* stream);

/* ---------------------------------------------------------------------------
 * The whole step in one call — [LLMC] §4's order: grad norm and clip scale,
 * the optional outlier check, then the AdamW + stochastic-rounding update of
 * the whole buffer [0, n). Enqueues mp_grad_norm's kernels, mp_outlier_check
 * (if outlier_state != NULL) and mp_adamw_step's kernel(s); same arguments,
 * same results as making those calls in that order with global_offset 0.
 * A small set (n <= 32,768, buffers vector-aligned, at most 32 decay
 * segments) runs as one thread-block cluster launch instead, with the same
 * results and the workspace left untouched. The first call on a device asks
 * the GPU whether it can run that cluster: make it before any stream
 * capture. (A ZeRO-1 shard calls the pieces: its norm must cover every
 * shard.)
 *
 *   grads        bf16[n], device. If host_grads is NULL, the gradients to use;
 *                otherwise it receives the device copy of host_grads.
 *   host_grads   bf16[n] in page-locked host memory (cudaHostAlloc'd or
 *                cudaHostRegister'ed), or NULL. The norm kernel reads it over
 *                the host link and writes `grads` in the same pass, so the
 *                transfer overlaps the reduction. MP_ERR_ACCESS if the device
 *                cannot read it.
 *   hyper        host struct: lr, beta1, beta2, eps, weight_decay, clip.
 *   workspace    as mp_grad_norm (mp_grad_norm_workspace_bytes(n) bytes).
 *   outlier_state, outlier_z, d_z   as mp_outlier_check's d_state, z_threshold
 *                and d_z; outlier_state NULL skips the check.
 *   d_norm, d_scale   float[1] device outputs (norm and clip scale).
 *   d_status     int32[1], device, may be NULL (as mp_adamw_step).
 *   host_norm    float[1] host destination of the norm (copied at the end of
 *                the stream's work; page-locked for an asynchronous copy), or
 *                NULL.
 * All other arguments as mp_adamw_step. Every argument is checked before
 * anything is enqueued.
 * Errors: as mp_grad_norm and mp_adamw_step, and MP_ERR_ACCESS.
 * ------------------------------------------------------------------------- */
int mp_optimizer_step(uint16_t* params, uint16_t* grads, const uint16_t* host_grads,
                      float* master, float* m, float* v, uint64_t n,
                      const mp_tensor_t* table, int32_t n_tensors,
                      const mp_hyper_t* hyper, int32_t t, uint32_t seed,
                      void* workspace, size_t workspace_bytes,
                      void* outlier_state, float outlier_z, double* d_z,
                      float* d_norm, float* d_scale, int32_t* d_status,
                      float* host_norm, void* stream);

/* ---------------------------------------------------------------------------
 * Host-to-device copy by the SMs — for gradients that arrive in page-locked
 * host memory. [LLMC] §3.3 hides transfers behind compute on a second
 * stream; here the transfer of the next step's gradients runs beside the
 * current step's update. The copy is a kernel of blocks_per_sm blocks of 256
 * threads per SM issuing 16-B loads of the host buffer over the host link;
 * with blocks_per_sm = 1 it fits beside the update kernel's resident blocks,
 * so the two run concurrently when launched on different streams.
 *
 *   dst            device memory, `bytes` bytes, written.
 *   host_src       page-locked host memory (cudaHostAlloc'd or
 *                  cudaHostRegister'ed) the device can read; read only; must
 *                  not change until the copy has run.
 *   bytes          any count; 0 is a no-op. Both pointers 16-B aligned take
 *                  the vector path; otherwise bytes are copied one by one.
 *   blocks_per_sm  1 .. 32.
 * Errors: MP_ERR_NULL, MP_ERR_RANGE, MP_ERR_ACCESS (host_src not page-locked
 *         or not device-visible), MP_ERR_CUDA.
 * ------------------------------------------------------------------------- */
int mp_copy_from_host(void* dst, const void* host_src, uint64_t bytes, int32_t blocks_per_sm, void* stream);

/* ---------------------------------------------------------------------------
 * Replayable steps: the step count on the device.
 *
 * mp_optimizer_step bakes t, seed and lr into its launches, so a recorded
 * launch sequence (a CUDA graph captured from a stream) would repeat one
 * step. mp_optimizer_step_graph reads them from device memory instead: the
 * norm's finalize kernel advances a device step counter and looks up that
 * step's bias corrections in a device table, and the update kernel reads
 * them from there. One capture then serves every later step, with no host
 * work per step. The arithmetic is mp_optimizer_step's: the same kernels'
 * per-element code, the same bias corrections (the table holds the values
 * the host computes for mp_adamw_step, [LLMC] §2.2 m_hat/v_hat and §4
 * t = step + 1; [CMU13] §1.7 the factor 1 - beta^t), so a run of graph steps
 * is bit-identical to the same run of mp_optimizer_step calls.
 *
 * The step state (device memory, 32 B, 16-B aligned, owned by the caller):
 *   t          steps taken so far (0 before the first). Each call adds 1 and
 *              updates with the new t. Set it to resume from a checkpoint.
 *   seed_base  step t rounds with seed = seed_base + t (mod 2^32).
 *   lr         learning rate of the next step; the caller may write it
 *              between steps (a schedule).
 *   seed, bc1, bc2   written by each call: the seed and bias corrections of
 *              the step it took.
 * ------------------------------------------------------------------------- */
typedef struct mp_step_state {
    int32_t t;
    uint32_t seed_base;
    float lr;
    uint32_t reserved0; /* 0 */
    uint32_t seed;
    float bc1, bc2;
    uint32_t reserved1; /* 0 */
} mp_step_state_t;

/* Length of the bias-correction table for (beta1, beta2): the first step t at
 * which both (float)(1 - beta^t) round to exactly 1.0f. Every later step has
 * the same corrections, so a table of this length serves every t. Returns 0
 * if beta1 or beta2 is outside [0, 1) or the length would exceed 2^26
 * entries (beta within ~2^-22 of 1). Host only; no CUDA call. */
int64_t mp_bias_table_len(float beta1, float beta2);

/* Fills out[2*(t-1)] = bc1(t), out[2*(t-1)+1] = bc2(t) for t = 1..len, with
 * bc(t) = (float)(1 - beta^t) computed in double exactly as mp_adamw_step's
 * host side does. `out` is HOST memory of 2*len floats; copy it to the
 * device for mp_optimizer_step_graph. Host only; no CUDA call.
 * Errors: MP_ERR_NULL, MP_ERR_RANGE (betas outside [0, 1), len < 1). */
int mp_bias_table(float beta1, float beta2, int64_t len, float* out);

/* ---------------------------------------------------------------------------
 * The whole step, replayable (see above). Enqueues the same kernels as
 * mp_optimizer_step; per call, on the device and in stream order:
 *   t = d_state->t + 1;  seed = d_state->seed_base + t;
 *   (bc1, bc2) = d_bias[min(t, bias_len) - 1];  lr = d_state->lr;
 *   then the norm, the optional outlier check and the update with those.
 * t advances on every call, also when the update is refused or skipped
 * (the train loop's step count moves on regardless, [LLMC] §4).
 *
 *   d_state      mp_step_state_t, device, 16-B aligned, read and written.
 *   d_bias       float[2*bias_len], device: mp_bias_table's contents for
 *                these betas; read only.
 *   bias_len     >= 1. If a step's t exceeds bias_len while the last entry
 *                is not (1.0f, 1.0f), or d_state->t is negative or already
 *                2^31 - 1, the step is refused on the device: nothing is
 *                written, t does not advance and *d_status gets MP_ERR_RANGE
 *                (if it held 0).
 *   hyper        as mp_optimizer_step; hyper->lr is not used (d_state->lr is).
 * Every other argument as mp_optimizer_step, and the same host-side checks.
 * Capture: make one call (a real step) before capturing, so the library's
 * per-device lookups are done; a capture records the pointers and n, so the
 * recorded graph must be replayed with those same buffers.
 * Errors: as mp_optimizer_step.
 * ------------------------------------------------------------------------- */
int mp_optimizer_step_graph(uint16_t* params, uint16_t* grads, const uint16_t* host_grads,
                            float* master, float* m, float* v, uint64_t n,
                            const mp_tensor_t* table, int32_t n_tensors,
                            const mp_hyper_t* hyper, mp_step_state_t* d_state,
                            const float* d_bias, int64_t bias_len,
                            void* workspace, size_t workspace_bytes,
                            void* outlier_state, float outlier_z, double* d_z,
                            float* d_norm, float* d_scale, int32_t* d_status,
                            float* host_norm, void* stream);

/* ---------------------------------------------------------------------------
 * Gradient norm without a workspace. The pages have no counterpart to this
 * call: it exists for callers that cannot allocate device memory — a host
 * framework that reserves all device memory in its own pool and hands a
 * plugin only its input and output buffers, or a loop that cannot afford the
 * device-wide synchronisation that cudaMalloc/cudaFree bring. It computes
 * exactly what mp_grad_norm computes, with the same kernels and the same
 * results, but keeps the per-block partial sums in a 32 KB scratch array the
 * library itself defines in device memory (room for 4096 partials; every GPU
 * that loads the library holds it until the process exits). Nothing is
 * allocated on any call, by the library or by anything it calls.
 *
 *   grads, n, clip, d_norm, d_scale, d_sumsq, stream: as for mp_grad_norm.
 *
 * The first call on a device looks up the scratch array's device address
 * (with that device current) and caches it; make that first call before any
 * stream capture. The cached address belongs to the device's primary
 * context: it assumes that context for the life of the process (no
 * cudaDeviceReset, no other driver context made current on that device).
 * Devices with an ordinal of 64 or more are looked up on every call. The
 * scratch is shared by all calls on a device and keeps
 * the last call's contents (each call overwrites every slot it reads, so
 * nothing needs clearing): calls that overlap on the GPU — on two streams,
 * or from two threads without ordering — race on it and must be serialised
 * by the caller.
 * Errors: as mp_grad_norm, and MP_ERR_WORKSPACE if the device would need more
 * than 4096 partials (a GPU with more than 1024 SMs; a 152-SM GB300 needs at
 * most 608).
 * ------------------------------------------------------------------------- */
int mp_grad_norm_noalloc(const uint16_t* grads, uint64_t n, float clip,
                         float* d_norm, float* d_scale, double* d_sumsq,
                         void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MP_ADAMW_H */
