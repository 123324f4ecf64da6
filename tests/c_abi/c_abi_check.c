/*
 * c_abi_check.c — drives libmpadamw.so from plain C (no Python, no PyTorch)
 * and checks the results against the CPU oracle compiled into the same
 * program. Test code: it allocates its own device buffers with cudaMalloc.
 *
 * One optimizer step (mp_optimizer_step, then a second call of the pieces:
 * mp_grad_norm + mp_adamw_step) on n = 100,003 elements split into 7 tensors
 * with alternating decay flags, against the oracle's own norm, clip scale
 * and steps; then mp_stochastic_round, mp_accumulate_sr and
 * mp_stochastic_round_fp16.
 * Then steps 3-6 as replayable steps: step 3 a plain mp_optimizer_step_graph
 * call, steps 4-6 replays of one CUDA graph captured from a stream, with
 * fresh gradients copied in between. Then the ZeRO-1 norm's two halves over
 * 4 shards, the learning-rate schedules and a host-to-device copy by the SMs.
 * Exit status 0 when every output is bit-identical to the oracle's (and the
 * copy to its source).
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "mp_adamw.h"
#include "mp_oracle.h"

#define N 100003u
#define NT 7

static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static uint32_t rng_u32(void) { /* xorshift64*: seeded synthetic inputs */
    rng_state ^= rng_state >> 12;
    rng_state ^= rng_state << 25;
    rng_state ^= rng_state >> 27;
    return (uint32_t)((rng_state * 0x2545F4914F6CDD1Dull) >> 32);
}
static float rng_uniform(void) { return (float)(rng_u32() >> 8) / 16777216.0f - 0.5f; }
static uint16_t to_bf16_bits(float x) { /* truncation: any bf16 pattern is a valid input */
    uint32_t u;
    memcpy(&u, &x, 4);
    return (uint16_t)(u >> 16);
}

#define CK(call) do { cudaError_t e_ = (call); if (e_ != cudaSuccess) { \
    fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_)); return 2; } } while (0)
#define MP(call) do { int s_ = (call); if (s_ != MP_OK) { \
    fprintf(stderr, "%s: %s\n", #call, mp_status_string(s_)); return 3; } } while (0)

static int same(const void* a, const void* b, size_t bytes, const char* what) {
    if (memcmp(a, b, bytes) != 0) {
        fprintf(stderr, "%s differs from the oracle\n", what);
        return 0;
    }
    return 1;
}

int main(void) {
    static uint16_t params[N], grads[N], params_o[N], out_sr[N], out_sr_o[N], out_h[N], out_h_o[N];
    static float master[N], m[N], v[N], master_o[N], m_o[N], v_o[N];
    for (uint32_t i = 0; i < N; ++i) {
        master[i] = 0.05f * rng_uniform();
        params[i] = to_bf16_bits(master[i]);
        grads[i] = to_bf16_bits(0.02f * rng_uniform());
        m[i] = 1e-3f * rng_uniform();
        v[i] = 1e-6f * (rng_uniform() + 0.5f);
    }
    mp_tensor_t table[NT];
    oracle_tensor otable[NT];
    uint64_t off = 0;
    for (int k = 0; k < NT; ++k) {
        uint64_t size = (k == NT - 1) ? N - off : (uint64_t)(N / NT + 17 * k);
        table[k].offset = off; table[k].size = size; table[k].decay = k % 2; table[k].reserved = 0;
        otable[k].offset = off; otable[k].size = size; otable[k].decay = k % 2; otable[k].pad = 0;
        off += size;
    }
    memcpy(params_o, params, sizeof params);
    memcpy(master_o, master, sizeof master);
    memcpy(m_o, m, sizeof m);
    memcpy(v_o, v, sizeof v);

    uint16_t *d_params, *d_grads, *d_sr, *d_h;
    float *d_master, *d_m, *d_v, *d_norm, *d_scale;
    int32_t* d_status;
    void* d_ws;
    const size_t ws_bytes = mp_grad_norm_workspace_bytes(N);
    CK(cudaMalloc((void**)&d_params, sizeof params));
    CK(cudaMalloc((void**)&d_grads, sizeof grads));
    CK(cudaMalloc((void**)&d_sr, sizeof out_sr));
    CK(cudaMalloc((void**)&d_h, sizeof out_h));
    CK(cudaMalloc((void**)&d_master, sizeof master));
    CK(cudaMalloc((void**)&d_m, sizeof m));
    CK(cudaMalloc((void**)&d_v, sizeof v));
    CK(cudaMalloc((void**)&d_norm, 4));
    CK(cudaMalloc((void**)&d_scale, 4));
    CK(cudaMalloc((void**)&d_status, 4));
    CK(cudaMalloc(&d_ws, ws_bytes));
    CK(cudaMemcpy(d_params, params, sizeof params, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_grads, grads, sizeof grads, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_master, master, sizeof master, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_m, m, sizeof m, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_v, v, sizeof v, cudaMemcpyHostToDevice));
    CK(cudaMemset(d_status, 0, 4));

    const mp_hyper_t hyper = {1e-3f, 0.9f, 0.95f, 1e-8f, 0.1f, 1.0f};
    /* step 1: the whole step in one call */
    MP(mp_optimizer_step(d_params, d_grads, NULL, d_master, d_m, d_v, N, table, NT, &hyper, 1, 11,
                         d_ws, ws_bytes, NULL, 0.0f, NULL, d_norm, d_scale, d_status, NULL, NULL));
    float norm1, scale1;
    CK(cudaMemcpy(&norm1, d_norm, 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(&scale1, d_scale, 4, cudaMemcpyDeviceToHost));
    /* step 2: the same through the separate calls */
    MP(mp_grad_norm(d_grads, N, hyper.clip, d_ws, ws_bytes, d_norm, d_scale, NULL, NULL));
    MP(mp_adamw_step(d_params, d_grads, d_master, d_m, d_v, 0, N, table, NT, hyper.lr, hyper.beta1, hyper.beta2,
                     hyper.eps, hyper.weight_decay, d_scale, 2, 12, d_status, NULL));
    float scale2;
    CK(cudaMemcpy(&scale2, d_scale, 4, cudaMemcpyDeviceToHost));
    /* standalone rounding of the new master, then accumulating the master into it */
    MP(mp_stochastic_round(d_sr, d_master, 0, N, 99, NULL));
    MP(mp_accumulate_sr(d_sr, d_master, 0, N, 98, NULL));
    MP(mp_stochastic_round_fp16(d_h, d_master, 0, N, 97, NULL));
    int32_t status;
    CK(cudaMemcpy(&status, d_status, 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(params, d_params, sizeof params, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(master, d_master, sizeof master, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(m, d_m, sizeof m, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(v, d_v, sizeof v, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out_sr, d_sr, sizeof out_sr, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out_h, d_h, sizeof out_h, cudaMemcpyDeviceToHost));

    /* the oracle's own chain: its norm and clip scale, then its steps. The GPU's
     * norm must be within 1e-6 of the oracle's fp64 one; the fp32 norms (and so
     * the scales) then agree except within ~1e-9 of a rounding boundary, and
     * the step is required to match bit for bit. */
    double sumsq;
    float norm_o, scale_o;
    oracle_grad_norm(grads, N, hyper.clip, &sumsq, &norm_o, &scale_o);
    if (!(fabs((double)norm1 - sqrt(sumsq)) <= 1e-6 * sqrt(sumsq)) || scale1 != scale_o || scale2 != scale_o) {
        fprintf(stderr, "norm %.9g scale %.9g/%.9g vs oracle %.9g %.9g\n", norm1, scale1, scale2, sqrt(sumsq),
                scale_o);
        return 1;
    }
    if (oracle_adamw_step(params_o, grads, master_o, m_o, v_o, 0, N, otable, NT, hyper.lr, hyper.beta1,
                          hyper.beta2, hyper.eps, hyper.weight_decay, scale_o, 1, 11) != 0 ||
        oracle_adamw_step(params_o, grads, master_o, m_o, v_o, 0, N, otable, NT, hyper.lr, hyper.beta1,
                          hyper.beta2, hyper.eps, hyper.weight_decay, scale_o, 2, 12) != 0)
        return 1;
    oracle_stochastic_round(out_sr_o, master_o, 0, N, 99);
    oracle_accumulate_sr(out_sr_o, master_o, 0, N, 98);
    oracle_stochastic_round_fp16(out_h_o, master_o, 0, N, 97);
    int ok = status == 0;
    ok &= same(params, params_o, sizeof params, "params");
    ok &= same(master, master_o, sizeof master, "master");
    ok &= same(m, m_o, sizeof m, "m");
    ok &= same(v, v_o, sizeof v, "v");
    ok &= same(out_sr, out_sr_o, sizeof out_sr, "stochastic round + accumulate");
    ok &= same(out_h, out_h_o, sizeof out_h, "fp16 stochastic round");

    /* steps 3..6 with the step count on the device: seed of step t = 10 + t */
    enum { FIRST = 3, LAST = 6 };
    static uint16_t grads_k[LAST - FIRST + 1][N];
    float scales[LAST - FIRST + 1];
    for (int k = 0; k <= LAST - FIRST; ++k)
        for (uint32_t i = 0; i < N; ++i) grads_k[k][i] = to_bf16_bits((0.01f + 0.01f * (float)k) * rng_uniform());
    const int64_t blen = mp_bias_table_len(hyper.beta1, hyper.beta2);
    float* bias = (float*)malloc(sizeof(float) * 2 * (size_t)blen);
    if (blen < 1 || bias == NULL) return 4;
    MP(mp_bias_table(hyper.beta1, hyper.beta2, blen, bias));
    float* d_bias;
    mp_step_state_t* d_state;
    CK(cudaMalloc((void**)&d_bias, sizeof(float) * 2 * (size_t)blen));
    CK(cudaMalloc((void**)&d_state, sizeof(mp_step_state_t)));
    CK(cudaMemcpy(d_bias, bias, sizeof(float) * 2 * (size_t)blen, cudaMemcpyHostToDevice));
    const mp_step_state_t state0 = {FIRST - 1, 10u, hyper.lr, 0u, 0u, 0.0f, 0.0f, 0u};
    CK(cudaMemcpy(d_state, &state0, sizeof state0, cudaMemcpyHostToDevice));
    cudaStream_t stream;
    CK(cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking));
    cudaGraph_t graph = NULL;
    cudaGraphExec_t exec = NULL;
    for (int t = FIRST; t <= LAST; ++t) {
        CK(cudaMemcpyAsync(d_grads, grads_k[t - FIRST], sizeof grads, cudaMemcpyHostToDevice, stream));
        if (t == FIRST) { /* a plain call, then the capture of the same call */
            MP(mp_optimizer_step_graph(d_params, d_grads, NULL, d_master, d_m, d_v, N, table, NT, &hyper, d_state,
                                       d_bias, blen, d_ws, ws_bytes, NULL, 0.0f, NULL, d_norm, d_scale, d_status,
                                       NULL, stream));
            CK(cudaStreamSynchronize(stream));
            CK(cudaStreamBeginCapture(stream, cudaStreamCaptureModeGlobal));
            MP(mp_optimizer_step_graph(d_params, d_grads, NULL, d_master, d_m, d_v, N, table, NT, &hyper, d_state,
                                       d_bias, blen, d_ws, ws_bytes, NULL, 0.0f, NULL, d_norm, d_scale, d_status,
                                       NULL, stream));
            CK(cudaStreamEndCapture(stream, &graph));
            CK(cudaGraphInstantiate(&exec, graph, 0));
        } else {
            CK(cudaGraphLaunch(exec, stream));
        }
        CK(cudaMemcpyAsync(&scales[t - FIRST], d_scale, 4, cudaMemcpyDeviceToHost, stream));
        CK(cudaStreamSynchronize(stream));
    }
    mp_step_state_t state;
    CK(cudaMemcpy(&state, d_state, sizeof state, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(&status, d_status, 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(params, d_params, sizeof params, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(master, d_master, sizeof master, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(m, d_m, sizeof m, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(v, d_v, sizeof v, cudaMemcpyDeviceToHost));
    for (int t = FIRST; t <= LAST; ++t) {
        oracle_grad_norm(grads_k[t - FIRST], N, hyper.clip, &sumsq, &norm_o, &scale_o);
        if (!(fabs((double)scale_o - (double)scales[t - FIRST]) <= 1e-6 * (double)scale_o)) {
            fprintf(stderr, "step %d: scale %.9g vs oracle %.9g\n", t, scales[t - FIRST], scale_o);
            return 1;
        }
        if (oracle_adamw_step(params_o, grads_k[t - FIRST], master_o, m_o, v_o, 0, N, otable, NT, hyper.lr,
                              hyper.beta1, hyper.beta2, hyper.eps, hyper.weight_decay, scales[t - FIRST], t,
                              10u + (uint32_t)t) != 0)
            return 1;
    }
    float bc1_o, bc2_o;
    oracle_bias_corrections(hyper.beta1, hyper.beta2, LAST, &bc1_o, &bc2_o);
    if (status != 0 || state.t != LAST || state.seed != 10u + LAST || state.bc1 != bc1_o || state.bc2 != bc2_o) {
        fprintf(stderr, "device step state t=%d seed=%u bc=(%.9g, %.9g), status %d\n", state.t, state.seed,
                state.bc1, state.bc2, status);
        ok = 0;
    }
    ok &= same(params, params_o, sizeof params, "params after graph steps");
    ok &= same(master, master_o, sizeof master, "master after graph steps");
    ok &= same(m, m_o, sizeof m, "m after graph steps");
    ok &= same(v, v_o, sizeof v, "v after graph steps");

    /* the ZeRO-1 norm in two halves: 4 shards' sums of squares, then the
     * scale from them in rank order; the oracle's ZeRO-1 norm of the same
     * sums must match bit for bit, and each sum the oracle's own to 1e-6 */
    enum { W = 4 };
    const uint32_t per = N / W; /* the last N % W elements are left out */
    double *d_parts, *d_total;
    double gpu_parts[W], total;
    CK(cudaMalloc((void**)&d_parts, sizeof gpu_parts));
    CK(cudaMalloc((void**)&d_total, sizeof total));
    CK(cudaMemcpy(d_grads, grads_k[0], sizeof grads, cudaMemcpyHostToDevice));
    for (int r = 0; r < W; ++r) MP(mp_grad_sumsq(d_grads + (size_t)r * per, per, d_ws, ws_bytes, d_parts + r, NULL));
    MP(mp_clip_scale_from_sumsq(d_parts, W, 0.25f, d_norm, d_scale, d_total, NULL));
    float zn, zs;
    CK(cudaMemcpy(gpu_parts, d_parts, sizeof gpu_parts, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(&total, d_total, sizeof total, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(&zn, d_norm, 4, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(&zs, d_scale, 4, cudaMemcpyDeviceToHost));
    double zsum_o;
    float zn_o, zs_o;
    oracle_norm_from_parts(gpu_parts, W, 0.25f, &zsum_o, &zn_o, &zs_o);
    if (total != zsum_o || zn != zn_o || zs != zs_o) {
        fprintf(stderr, "ZeRO-1 norm %.9g scale %.9g vs oracle %.9g %.9g\n", zn, zs, zn_o, zs_o);
        ok = 0;
    }
    for (int r = 0; r < W; ++r) {
        const double ref = oracle_sumsq(grads_k[0] + (size_t)r * per, per);
        if (!(fabs(gpu_parts[r] - ref) <= 1e-6 * ref)) {
            fprintf(stderr, "shard %d sum of squares %.17g vs oracle %.17g\n", r, gpu_parts[r], ref);
            ok = 0;
        }
    }
    cudaFree(d_parts);
    cudaFree(d_total);

    /* learning-rate schedules (host only): every step of four runs */
    for (int kind = MP_LR_CONSTANT; kind <= MP_LR_WSD; ++kind) {
        const mp_lr_schedule_t sch = {kind, 0, 50, 1000, 6e-4f, 6e-5f, 0.2f, 0.0f};
        for (int64_t t = 1; t <= 1100; ++t) {
            float lr;
            MP(mp_lr_at(&sch, t, &lr));
            const float lr_o = oracle_lr(kind, 50, 1000, 6e-4f, 6e-5f, 0.2f, t);
            if (memcmp(&lr, &lr_o, 4) != 0) {
                fprintf(stderr, "schedule %d step %lld: lr %.9g vs oracle %.9g\n", kind, (long long)t, lr, lr_o);
                ok = 0;
                break;
            }
        }
    }

    /* a host-to-device copy by the SMs from page-locked memory */
    uint16_t* h_pinned;
    CK(cudaHostAlloc((void**)&h_pinned, sizeof grads, cudaHostAllocDefault));
    memcpy(h_pinned, grads_k[1], sizeof grads);
    CK(cudaMemset(d_grads, 0, sizeof grads));
    MP(mp_copy_from_host(d_grads, h_pinned, sizeof grads, 1, NULL));
    CK(cudaMemcpy(grads, d_grads, sizeof grads, cudaMemcpyDeviceToHost));
    ok &= same(grads, grads_k[1], sizeof grads, "host-to-device copy by the SMs");
    cudaFreeHost(h_pinned);
    printf("c_abi_check: %s (n=%u, norm %.7g, scale %.7g; graph steps %d-%d)\n",
           ok ? "bit-identical to the oracle" : "MISMATCH", N, norm1, scale1, FIRST, LAST);
    cudaGraphExecDestroy(exec); cudaGraphDestroy(graph); cudaStreamDestroy(stream); free(bias);
    cudaFree(d_bias); cudaFree(d_state);
    cudaFree(d_params); cudaFree(d_grads); cudaFree(d_sr); cudaFree(d_h); cudaFree(d_master); cudaFree(d_m); cudaFree(d_v);
    cudaFree(d_norm); cudaFree(d_scale); cudaFree(d_status); cudaFree(d_ws);
    return ok ? 0 : 1;
}
