"""Benchmark of the mixed-precision optimizer step on GB300.

One step = the whole hot path over the Llama-3-8B parameter set (8,030,261,248
params, 291 tensors, one flat buffer, about 128 GB of optimizer state in HBM):
global grad norm + clip scale (mp_grad_norm: two kernels) and the fused
AdamW + stochastic-rounding step with fp32 master weights (mp_adamw_step: 40
launches of about 200M elements). Inputs are synthetic and already resident in
HBM; the 241 GB touched per step are far larger than the 129 MB L2, so no
flush is needed between steps.

Prints ONE JSON line (rank 0). Also reports: the roofline of the dominant
kernel (the step kernel, 28 algorithmic bytes per parameter, timed over 16 or
more event-bracketed steps after the timed region) against the measured HBM
copy bandwidth, with its DRAM traffic scaled from a committed ncu capture;
the other path variants (no-master step, norm, standalone roundings, 8 ZeRO-1
shard launches; the GPT-2 1.5B set whole and as 8 shards; the
stochastic-rounding stress set: kernel throughput and 1000-step drift); an
end-to-end number through the C ABI with the gradients copied from pinned
host memory every step; SM clocks sampled during the timed region; and the
CPU oracle timed on a bounded sample as a reported baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload tiny|gpt2_124m|gpt2_1558m|llama3_8b]
With N > 1 (launched by torch.distributed.run) the ranks run the ZeRO-1 step
(zero1.py): reduce-scatter of the gradients, each rank's shard of the norm and
the update, all-gather of the bf16 weights; the time is the max over ranks.
--replicas runs an independent single-GPU step per rank instead.
"""
import argparse
import hashlib
import json
import os
import platform
import re
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "AdamW+SR step: Gparams/s and HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "Gparams/s"
WORKLOAD = "llama3_8b"  # the default line; --workload picks the other parameter sets
WORKLOAD_NAMES = {
    "tiny": "tiny GPT-style parameter set (d 32, 2 layers, 28,672 params)",
    "gpt2_124m": "GPT-2 124M parameter set (V 50304, T 1024, d 768, 12 layers, tied wte)",
    "gpt2_1558m": "GPT-2 1.5B parameter set (V 50304, T 1024, d 1600, 48 layers, tied wte)",
    "llama3_8b": "Llama-3-8B parameter set (d 4096, 32 layers, GQA 32/8, SwiGLU 14336, V 128256 untied)",
}
STEP_BYTES_MASTER = 28   # 2 grad + 3x4 (master, m, v) read; 3x4 + 2 (param) written
STEP_BYTES_NOMASTER = 22
NORM_BYTES = 2
SR_BYTES = 6
ACC_BYTES = 8  # accumulate: read bf16 + fp32, write bf16
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal (context only)
STEP_KERNEL_SOURCES = ["mixed_precision_adamw_gb300/csrc/mp_step.cu",
                       "mixed_precision_adamw_gb300/csrc/mp_step.cuh",
                       "mixed_precision_adamw_gb300/csrc/mp_device.cuh",
                       "mixed_precision_adamw_gb300/csrc/mp_tma.cuh"]
# The library runs a step launch through its TMA-staged kernel (one block per
# SM, tiles of 2304 elements with master) when the launch holds at least two
# tiles per SM; shorter launches take the register kernel. Used for labels only.
TMA_TILE_MASTER = 2304
TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "adamw_step_traffic.json")
KERNEL_SAMPLES = 16  # event-bracketed step calls after the timed region, at least


# ---------------------------------------------------------------------------
# distributed plumbing (timing only)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    """Max of a per-rank scalar (the step time) over all ranks."""
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(params_per_rank: int, world: int, steps: int, max_seconds: float) -> float:
    """Gparams/s over all ranks: every rank updates params_per_rank per step."""
    return params_per_rank * world * steps / max_seconds / 1e9


# ---------------------------------------------------------------------------
# measurement helpers
# ---------------------------------------------------------------------------
def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def step_kernel_name(launch_elems: float, device) -> str:
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    tma = launch_elems >= 2 * sms * TMA_TILE_MASTER + 64
    return "adamw_tma_kernel<master>" if tma else "adamw_vec_kernel<master>"


def kernel_source_hash() -> str:
    """Hash of the step kernel's code with comments and blank space removed,
    so that editing a comment does not invalidate recorded counters."""
    h = hashlib.sha256()
    for rel in STEP_KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = "\n".join(line.strip() for line in text.splitlines() if line.strip())
        h.update(text.encode())
    return h.hexdigest()[:16]


def profiled_traffic_bytes(launch_elems: float):
    """DRAM bytes (read + write) of one step-kernel launch of `launch_elems`
    elements, from the committed ncu capture whose launch size is closest,
    scaled by elements (the kernel streams each element once), if that
    capture was taken on the current kernel source; else None."""
    try:
        with open(TRAFFIC_PROFILE) as f:
            prof = json.load(f)
    except (OSError, ValueError):
        return None, None
    current = kernel_source_hash()
    caps = [c for c in prof.get("captures", []) if c.get("kernel_source_sha256_16") == current]
    if not caps:
        return None, None
    cap = min(caps, key=lambda c: abs(c["launch_elems"] - launch_elems))
    per_elem = (cap["dram_bytes_read"] + cap["dram_bytes_write"]) / cap["launch_elems"]
    return int(round(per_elem * launch_elems)), cap["launch_elems"]


class ClockSampler:
    """nvidia-smi clock/throttle samples every 100 ms during the timed regions."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.path = None
        self.gpu = gpu_index
        if shutil.which("nvidia-smi") is None:
            return
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        self.fh = open(self.path, "w")
        self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.QUERY}",
                                      "--format=csv,noheader,nounits", "-lms", "100"],
                                     stdout=self.fh, stderr=subprocess.DEVNULL)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args, world, rank, local):
    import mixed_precision_adamw_gb300 as mp
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    H = W.HYPER
    workload = args.workload
    entries = W.layout(W.specs_for(workload))
    if args.params:
        entries = prefix_entries(entries, args.params)
    tab = W.table(entries)
    N = W.total(entries)
    st = W.make_state(workload, device=device, entries=entries)
    grads = [W.make_grads(workload, s, device=device, entries=entries) for s in (1, 2)]
    opt = mp.Optimizer(tab, lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"],
                       weight_decay=H["weight_decay"], clip=H["clip"], device=device)
    stream = torch.cuda.current_stream(device)
    kw = dict(lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"], weight_decay=H["weight_decay"])
    step_no = [0]

    def one_step(ev_pair=None):
        step_no[0] += 1
        t = step_no[0]
        g = grads[t % 2]
        mp.mp_grad_norm(g, H["clip"], opt.workspace, opt.d_norm, opt.d_scale, n=N, stream=stream)
        if ev_pair is not None:
            ev_pair[0].record(stream)
        mp.mp_adamw_step(st["params"], g, st["master"], st["m"], st["v"], opt.table, d_grad_scale=opt.d_scale,
                         t=t, seed=W.step_seed(t), d_status=opt.d_status, n=N, stream=stream, **kw)
        if ev_pair is not None:
            ev_pair[1].record(stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    barrier(world)

    # The timed region: K chained steps (the kernels of consecutive steps
    # follow each other with programmatic dependent launch; no event sits
    # between them).
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    torch.cuda.synchronize()
    barrier(world)
    start.record(stream)
    for _ in range(args.steps):
        one_step()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    total_ms = start.elapsed_time(end)
    opt.check_status()
    max_s = max_over_ranks(total_ms / 1e3, world, device)
    value = whole_job_value(N, world, args.steps, max_s)
    ms_per_step = max_s * 1e3 / args.steps

    # The step kernel alone: events around the update of each of
    # KERNEL_SAMPLES further steps (norm, event, update, event), so the
    # sample count does not depend on --steps. A step's update is one or more
    # launches of the same kernel (ranges above 201,326,592 elements are cut
    # into near-equal launches); the events bracket all of them.
    launches = len(mp.mp_step_launches(0, N, opt.table))
    samples = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(max(KERNEL_SAMPLES, args.kernel_samples))]
    for ev in samples:
        one_step(ev)
    torch.cuda.synchronize()
    clocks = sampler.stop()  # sampled over both timed regions
    opt.check_status()
    step_call_ms = [a.elapsed_time(b) for a, b in samples]
    step_kernel_ms = statistics.mean(step_call_ms)

    peak, peak_kind = measured_hbm_peak()
    achieved = STEP_BYTES_MASTER * N / (step_kernel_ms / 1e3) / 1e9
    traffic, traffic_from = profiled_traffic_bytes(N / launches) if not args.params else (None, None)
    roofline = {"bound": "hbm", "kernel": step_kernel_name(N / launches, device), "achieved": round(achieved, 1),
                "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                "traffic": traffic,
                "traffic_source": (f"ncu capture of a {traffic_from}-element launch (profiles/adamw_step_traffic.json), "
                                   f"scaled by elements to this workload's launches" if traffic else None),
                "algorithmic_bytes_per_launch": round(STEP_BYTES_MASTER * N / launches),
                "launches_per_step": launches,
                "kernel_ms_per_launch": round(step_kernel_ms / launches, 5),
                "kernel_ms_per_step": round(step_kernel_ms, 5), "kernel_ms_samples": len(samples),
                "kernel_ms_per_step_median": round(statistics.median(step_call_ms), 5),
                "kernel_ms_per_step_min": round(min(step_call_ms), 5),
                "how": "achieved = 28 B x params / mean CUDA-event time of a step's update launches "
                       "(= algorithmic bytes per launch / mean launch duration)"}

    roofline["frac_of_nominal"] = round(achieved / NOMINAL_HBM_GBS, 4)
    if args.quick:
        variants, e2e = None, None
    else:
        ceiling = copy_ceiling(STEP_BYTES_MASTER // 2 * N, stream, device)
        ceiling["step_kernel_frac"] = round(achieved / ceiling["gbs"], 4)
        roofline["copy_ceiling"] = ceiling
        variants = measure_variants(mp, st, grads[0], opt, N, entries, tab, stream, device, peak)
        e2e = measure_e2e(mp, st, grads[0], opt, N, stream, device, kw, min(args.steps, 200), step_no)
        # last: the probes overwrite the bf16 weights
        probes = measure_stream_probes(st, grads[0], N, stream, peak)
        best = max(v["gbs"] for k, v in probes.items() if k.startswith("step_streams"))
        probes["step_kernel_frac_of_best_step_streams"] = round(achieved / best, 4)
        roofline["sm_stream_probes"] = probes

    if rank != 0:
        return None
    # norm partials + norm finalize + the step's launches, as the library splits them
    launches_per_step = 2 + launches
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAMES[workload],
                   "params": N, "tensors": len(entries), "variant": "fp32 master + bf16 params, clip 1.0",
                   "bytes_per_param": STEP_BYTES_MASTER + NORM_BYTES,
                   "l2": (f"no flush: {(STEP_BYTES_MASTER + NORM_BYTES) * N / 1e9:.2f} GB touched per step, > 129 MB L2"
                          if (STEP_BYTES_MASTER + NORM_BYTES) * N > 4 * 129e6 else
                          "working set L2-resident (launch-bound latency case)"),
                   "parallelism": f"replicas{world}" if world > 1 else "single GPU"},
        "hbm_gbs": round((STEP_BYTES_MASTER + NORM_BYTES) * N * args.steps / (total_ms / 1e3) / 1e9, 1),
        "hbm_frac_of_measured": round((STEP_BYTES_MASTER + NORM_BYTES) * N * args.steps / (total_ms / 1e3)
                                      / 1e9 / peak, 4),
        "roofline": roofline, "variants": variants, "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
    }
    if args.params:
        line["config"]["workload"] += f", first {N} params only"
    if not args.quick:
        # other parameter sets, after this one's state is released
        del st, grads, opt
        torch.cuda.empty_cache()
        if workload == WORKLOAD and not args.params:
            line["variants"]["gpt2_1558m_whole_vs_8_shards"] = measure_shards_1558m(mp, stream, device, peak)
        line["variants"]["sr_stress"] = measure_sr_stress(mp, stream, device, peak)
    if world == 1 and not args.no_cpu_baseline and not args.quick:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds, workload)
    return line


def run_zero1(args, world, rank, local):
    """The ZeRO-1 step over `world` ranks (llm.c ch. 04 §3.2-§3.3, §4):
    reduce-scatter of the gradients, the shard's share of the norm,
    all-gather of the per-rank sums, the shard update, all-gather of the
    bf16 weights. The whole model's parameters are updated once per step
    across all ranks, so the value is params x steps / the slowest rank's
    time (strong scaling: the work per step does not grow with N)."""
    import mixed_precision_adamw_gb300 as mp
    from mixed_precision_adamw_gb300.zero1 import Zero1Optimizer
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if not torch.distributed.is_initialized():
        if world == 1:  # a one-rank group outside torchrun (--zero1)
            import socket
            with socket.socket() as sk:
                sk.bind(("127.0.0.1", 0))
                port = sk.getsockname()[1]
            for k, v in (("MASTER_ADDR", "127.0.0.1"), ("MASTER_PORT", str(port)), ("RANK", "0"),
                         ("WORLD_SIZE", "1")):
                os.environ.setdefault(k, v)
        torch.distributed.init_process_group(backend="nccl")
    H = W.HYPER
    workload = args.workload
    entries = W.layout(W.specs_for(workload))
    if args.params:
        entries = prefix_entries(entries, args.params)
    tab = W.table(entries)
    N = W.total(entries)
    zopt = Zero1Optimizer(tab, lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"],
                          weight_decay=H["weight_decay"], clip=H["clip"], device=device)
    per = zopt.layout.size
    st = W.make_state(workload, device=device, entries=entries)
    params = st["params"]
    shard = zopt.make_shard_state(st["master"])
    del st
    torch.cuda.empty_cache()
    # each rank's backward pass gives its own gradients: seeded by rank
    grads = [W.make_grads(workload, s, device=device, entries=entries, seed=W.BASE_SEED + 7919 * rank)
             for s in (1, 2)]
    stream = torch.cuda.current_stream(device)
    step_no = [0]

    def one_step(g=None):
        step_no[0] += 1
        t = step_no[0]
        zopt.step(params, grads[t % 2] if g is None else g, shard["master"], shard["m"], shard["v"], t,
                  W.step_seed(t), stream=stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    barrier(world)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    barrier(world)
    start.record(stream)
    for _ in range(args.steps):
        one_step()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    total_ms = start.elapsed_time(end)
    assert zopt.take_status() == 0
    max_s = max_over_ranks(total_ms / 1e3, world, device)
    value = N * args.steps / max_s / 1e9
    ms_per_step = max_s * 1e3 / args.steps

    # the shard update alone (the dominant kernel), after the timed region
    kw = dict(lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"], weight_decay=H["weight_decay"])
    sl = zopt.layout.slice()
    ms = time_events(lambda: mp.mp_adamw_step(params[sl], zopt.grad_shard, shard["master"], shard["m"],
                                              shard["v"], zopt.table, d_grad_scale=zopt.d_scale, t=step_no[0],
                                              seed=1, global_offset=zopt.layout.offset, n=per, stream=stream, **kw),
                     max(KERNEL_SAMPLES, args.kernel_samples), stream)
    launches = len(mp.mp_step_launches(zopt.layout.offset, per, zopt.table))
    peak, peak_kind = measured_hbm_peak()
    achieved = STEP_BYTES_MASTER * per / ms / 1e6
    traffic, traffic_from = profiled_traffic_bytes(per / launches) if not args.params else (None, None)
    roofline = {"bound": "hbm", "kernel": step_kernel_name(per / launches, device) + " (this rank's shard)",
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "peak_kind": peak_kind, "traffic": traffic,
                "algorithmic_bytes_per_launch": round(STEP_BYTES_MASTER * per / launches),
                "launches_per_step": launches, "kernel_ms_per_step": round(ms, 5),
                "kernel_ms_samples": LAST_TIMING["launches"]}
    e2e = None
    if not args.quick:
        # end to end: this rank's gradients from pinned host memory, the
        # norm read back every step
        host_g = torch.empty(N, dtype=torch.bfloat16, pin_memory=True)
        host_g.copy_(grads[0])
        dev_g = grads[1]
        host_norm = torch.empty(1, dtype=torch.float32, pin_memory=True)
        iters = min(args.steps, 50)

        def e2e_step():
            mp.mp_copy_from_host(dev_g, host_g, stream=stream)  # the SMs read the pinned gradients
            one_step(dev_g)
            host_norm.copy_(zopt.d_norm, non_blocking=True)
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(iters):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e_s = max_over_ranks(a.elapsed_time(b) / 1e3, world, device)
        e2e = {"value": round(N * iters / e_s / 1e9, 3), "unit": UNIT, "h2d_bytes_per_step": 2 * N,
               "d2h_bytes_per_step": 4, "steps": iters,
               "api": "mp_copy_from_host + Zero1Optimizer.step (per rank: gradients copied from pinned host "
                      "memory first)"}
    if rank != 0:
        return None
    return {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAMES[workload] + (f", first {N} params only" if args.params else ""),
                   "params": N, "shard_params": per, "tensors": len(entries),
                   "variant": "fp32 master + bf16 params, clip 1.0",
                   "l2": f"no flush: {30 * per / 1e9:.2f} GB of optimizer traffic per rank per step, > 129 MB L2",
                   "parallelism": f"zero1 dp{world} (NCCL reduce-scatter avg, all-gather)"},
        "roofline": roofline, "e2e": e2e, "clocks": clocks,
        # per step: norm partials + sums-only finalize + scale + the shard's launches
        "gpu_launches": (3 + launches) * args.steps,
    }


LAST_TIMING = {}


def time_events(fn, iters, stream):
    """Mean CUDA-event time of fn over `iters` launches after one warm-up;
    the median and minimum are left in LAST_TIMING."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    fn()
    torch.cuda.synchronize()
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) for a, b in evs]
    LAST_TIMING.clear()
    LAST_TIMING.update(ms_median=round(statistics.median(times), 5), ms_min=round(min(times), 5), launches=iters)
    return statistics.mean(times)


def copy_ceiling(nbytes, stream, device, cap=1 << 32):
    """A plain device-to-device copy (cudaMemcpyAsync, through torch's
    copy_) moving as many bytes as the step kernel reads and writes, or 4 GiB
    each way at most: the practical ceiling of a stream that reads and writes
    equal amounts."""
    nbytes = min(nbytes, cap) // 16 * 16
    src = torch.empty(nbytes, dtype=torch.uint8, device=device)
    dst = torch.empty_like(src)
    src.fill_(1)
    ms = time_events(lambda: dst.copy_(src), 10, stream)
    del src, dst
    return {"gbs": round(2 * nbytes / ms / 1e6, 1), "bytes_each_way": nbytes,
            "what": "device-to-device cudaMemcpyAsync, CUDA-event mean of 10"}


def measure_variants(mp, st, g, opt, N, entries, tab, stream, device, peak):
    H = W.HYPER
    kw = dict(lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"], weight_decay=H["weight_decay"])
    out = {}
    iters = 20
    ms = time_events(lambda: mp.mp_grad_norm(g, H["clip"], opt.workspace, opt.d_norm, opt.d_scale, n=N,
                                             stream=stream), iters, stream)
    out["grad_norm"] = {**LAST_TIMING, "ms": round(ms, 5), "gbs": round(NORM_BYTES * N / ms / 1e6, 1),
                        "frac": round(NORM_BYTES * N / ms / 1e6 / peak, 4), "bytes_per_param": NORM_BYTES}
    # no-master variant, in place on params, m, v (no extra copy: the
    # Llama-3-8B state alone is 128 GB)
    ms = time_events(lambda: mp.mp_adamw_step(st["params"], g, None, st["m"], st["v"], opt.table,
                                              d_grad_scale=opt.d_scale, t=5, seed=5, n=N, stream=stream, **kw),
                     iters, stream)
    out["step_no_master"] = {**LAST_TIMING, "ms": round(ms, 5), "gparams_s": round(N / ms / 1e6, 2),
                             "gbs": round(STEP_BYTES_NOMASTER * N / ms / 1e6, 1),
                             "frac": round(STEP_BYTES_NOMASTER * N / ms / 1e6 / peak, 4),
                             "bytes_per_param": STEP_BYTES_NOMASTER}
    ms = time_events(lambda: mp.mp_stochastic_round(st["params"], st["master"], 7, n=N, stream=stream), iters,
                     stream)
    out["stochastic_round"] = {**LAST_TIMING, "ms": round(ms, 5), "gelems_s": round(N / ms / 1e6, 2),
                               "gbs": round(SR_BYTES * N / ms / 1e6, 1),
                               "frac": round(SR_BYTES * N / ms / 1e6 / peak, 4), "bytes_per_elem": SR_BYTES}
    # the same rounding onto fp16's grid (into the params buffer, viewed as fp16)
    h16 = st["params"].view(torch.float16)
    ms = time_events(lambda: mp.mp_stochastic_round_fp16(h16, st["master"], 7, n=N, stream=stream), iters,
                     stream)
    out["stochastic_round_fp16"] = {**LAST_TIMING, "ms": round(ms, 5), "gelems_s": round(N / ms / 1e6, 2),
                                    "gbs": round(SR_BYTES * N / ms / 1e6, 1),
                                    "frac": round(SR_BYTES * N / ms / 1e6 / peak, 4), "bytes_per_elem": SR_BYTES}
    # bf16 accumulation with stochastic rounding (params += master, in place)
    ms = time_events(lambda: mp.mp_accumulate_sr(st["params"], st["master"], 9, n=N, stream=stream), iters,
                     stream)
    out["accumulate_sr"] = {**LAST_TIMING, "ms": round(ms, 5), "gelems_s": round(N / ms / 1e6, 2),
                            "gbs": round(ACC_BYTES * N / ms / 1e6, 1),
                            "frac": round(ACC_BYTES * N / ms / 1e6 / peak, 4), "bytes_per_elem": ACC_BYTES}
    per = N // 8

    def shards():
        for r in range(8):
            sl = slice(r * per, (r + 1) * per)
            mp.mp_adamw_step(st["params"][sl], g[sl], st["master"][sl], st["m"][sl], st["v"][sl], opt.table,
                             d_grad_scale=opt.d_scale, t=6, seed=6, global_offset=r * per, n=per, stream=stream,
                             **kw)
    ms = time_events(shards, iters // 2, stream)
    out["step_8_shards"] = {**LAST_TIMING, "ms": round(ms, 5), "gparams_s": round(N / ms / 1e6, 2),
                            "gbs": round(STEP_BYTES_MASTER * N / ms / 1e6, 1), "launches": 8}
    return out


def measure_stream_probes(st, g, N, stream, peak):
    """Compute-free probes (libmpprobe.so, measurement only): the step's five
    streams with its tiling, vector widths, cache hints and occupancy, values
    written back unchanged; and a plain 16-B vector copy of 4 GiB. They give
    the practical ceiling of kernels on the SMs for this read/write mix,
    beside the copy engines' figure (copy_ceiling)."""
    import ctypes
    lib = ctypes.CDLL(os.path.join(ROOT, "mixed_precision_adamw_gb300", "libmpprobe.so"))
    vp, u64, i32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int
    lib.mp_probe_step_streams.argtypes = [vp, vp, vp, vp, vp, u64, i32, vp]
    lib.mp_probe_copy.argtypes = [vp, vp, u64, i32, vp]
    lib.mp_probe_step_streams_bulk.argtypes = [vp, vp, vp, vp, vp, u64, i32, i32, i32, vp, vp]
    lib.mp_probe_step_streams_bulk_tile.argtypes = [vp, vp, vp, vp, vp, u64, ctypes.c_uint32, i32, i32, i32, vp, vp]
    lib.mp_probe_copy_bulk.argtypes = [vp, vp, u64, i32, i32, i32, vp, vp]
    err = torch.zeros(1, dtype=torch.int32, device=g.device)
    chunk = 201_326_592  # the step's launch size on the large sets (whole 2048-element tiles)
    n = N // 2048 * 2048
    out = {}
    for bps in (3, 4, 8):
        def run():
            for a in range(0, n, chunk):
                b = min(n, a + chunk)
                rc = lib.mp_probe_step_streams(st["params"][a:].data_ptr(), g[a:].data_ptr(),
                                               st["master"][a:].data_ptr(), st["m"][a:].data_ptr(),
                                               st["v"][a:].data_ptr(), b - a, bps, stream.cuda_stream)
                assert rc == 0, rc
        ms = time_events(run, 5, stream)
        out[f"step_streams_{bps}_blocks_per_sm"] = {"gbs": round(STEP_BYTES_MASTER * n / ms / 1e6, 1),
                                                    "frac": round(STEP_BYTES_MASTER * n / ms / 1e6 / peak, 4),
                                                    "ms": round(ms, 5)}
    # the same streams staged through shared memory by TMA bulk copies
    for bps, stages, hint in ((1, 3, 1), (1, 3, 0), (1, 4, 1), (1, 7, 1), (2, 2, 1), (2, 3, 1)):
        def run_bulk():
            for a in range(0, n, chunk):
                b = min(n, a + chunk)
                rc = lib.mp_probe_step_streams_bulk(st["params"][a:].data_ptr(), g[a:].data_ptr(),
                                                    st["master"][a:].data_ptr(), st["m"][a:].data_ptr(),
                                                    st["v"][a:].data_ptr(), b - a, bps, stages, hint,
                                                    err.data_ptr(), stream.cuda_stream)
                assert rc == 0, rc
        ms = time_events(run_bulk, 5, stream)
        key = f"step_streams_tma_bulk_{bps}_blocks_per_sm_{stages}_stages" + ("_evict_first" if hint else "")
        out[key] = {"gbs": round(STEP_BYTES_MASTER * n / ms / 1e6, 1),
                    "frac": round(STEP_BYTES_MASTER * n / ms / 1e6 / peak, 4), "ms": round(ms, 5)}
    # larger tiles with one tile of loads in flight per SM (launches stay multiples of the tile)
    for tile in (6144, 8192):
        nt = N // tile * tile
        if nt == 0:
            continue
        def run_bulk_tile():
            for a in range(0, nt, chunk):
                b = min(nt, a + chunk)
                rc = lib.mp_probe_step_streams_bulk_tile(st["params"][a:].data_ptr(), g[a:].data_ptr(),
                                                         st["master"][a:].data_ptr(), st["m"][a:].data_ptr(),
                                                         st["v"][a:].data_ptr(), b - a, tile, 1, 2, 1,
                                                         err.data_ptr(), stream.cuda_stream)
                assert rc == 0, rc
        ms = time_events(run_bulk_tile, 5, stream)
        out[f"step_streams_tma_bulk_{tile}_tiles_1_blocks_per_sm_2_stages_evict_first"] = {
            "gbs": round(STEP_BYTES_MASTER * nt / ms / 1e6, 1),
            "frac": round(STEP_BYTES_MASTER * nt / ms / 1e6 / peak, 4), "ms": round(ms, 5)}
    nbytes = min(STEP_BYTES_MASTER // 2 * N, 1 << 32) // 16 * 16
    src = torch.empty(nbytes, dtype=torch.uint8, device=g.device)
    dst = torch.empty_like(src)
    src.fill_(1)
    for bps in (4, 8):
        ms = time_events(lambda: lib.mp_probe_copy(dst.data_ptr(), src.data_ptr(), nbytes // 16, bps,
                                                   stream.cuda_stream), 10, stream)
        out[f"copy_16B_{bps}_blocks_per_sm"] = {"gbs": round(2 * nbytes / ms / 1e6, 1),
                                                "frac": round(2 * nbytes / ms / 1e6 / peak, 4), "ms": round(ms, 5)}
    tile_bytes = 2048 * 14
    tiles = nbytes // tile_bytes
    for bps, stages, hint in ((1, 7, 1), (2, 3, 1)):
        def run_copy_bulk():
            rc = lib.mp_probe_copy_bulk(dst.data_ptr(), src.data_ptr(), tiles, bps, stages, hint, err.data_ptr(),
                                        stream.cuda_stream)
            assert rc == 0, rc
        ms = time_events(run_copy_bulk, 10, stream)
        gbs = 2 * tiles * tile_bytes / ms / 1e6
        out[f"copy_tma_bulk_{bps}_blocks_per_sm_{stages}_stages_evict_first"] = {
            "gbs": round(gbs, 1), "frac": round(gbs / peak, 4), "ms": round(ms, 5)}
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError("a TMA bulk probe gave up waiting on its mbarrier")
    del src, dst
    out["what"] = ("compute-free SM kernels: the step's streams (28 B/param, written back unchanged) in "
                   f"launches of {chunk} params, through registers and through TMA bulk copies staged in "
                   f"shared memory (one issuing thread per block, stages of 2048-param tiles (28 KB) or of "
                   f"6144 and 8192 params); a 16-B copy of {nbytes} bytes "
                   "and a TMA bulk copy of its whole 28 KB tiles")
    return out


def measure_shards_1558m(mp, stream, device, peak):
    """The GPT-2 1.5B set (1,557,686,400 params): one whole-buffer step
    against the same step as 8 contiguous shard launches of 194,710,800
    params each (the ZeRO-1 layout on one GPU, no communication). The tests
    check that both give the same bits."""
    H = W.HYPER
    name = "gpt2_1558m"
    entries = W.layout(W.specs_for(name))
    tab = W.table(entries)
    N = W.total(entries)
    st = W.make_state(name, device=device)
    g = W.make_grads(name, 1, device=device)
    opt = mp.Optimizer(tab, lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"],
                       weight_decay=H["weight_decay"], clip=H["clip"], device=device)
    kw = dict(lr=H["lr"], beta1=H["beta1"], beta2=H["beta2"], eps=H["eps"], weight_decay=H["weight_decay"],
              d_grad_scale=opt.d_scale, stream=stream)
    mp.mp_grad_norm(g, H["clip"], opt.workspace, opt.d_norm, opt.d_scale, n=N, stream=stream)
    per = N // 8
    ms_whole = time_events(lambda: mp.mp_adamw_step(st["params"], g, st["master"], st["m"], st["v"], opt.table,
                                                    t=1, seed=W.step_seed(1), n=N, **kw), 10, stream)
    whole = dict(LAST_TIMING)

    def shards():
        for r in range(8):
            sl = slice(r * per, (r + 1) * per)
            mp.mp_adamw_step(st["params"][sl], g[sl], st["master"][sl], st["m"][sl], st["v"][sl], opt.table,
                             t=1, seed=W.step_seed(1), global_offset=r * per, n=per, **kw)
    ms_sh = time_events(shards, 10, stream)
    out = {"params": N, "shard_params": per,
           "whole": {**whole, "ms": round(ms_whole, 5), "gparams_s": round(N / ms_whole / 1e6, 2),
                     "gbs": round(STEP_BYTES_MASTER * N / ms_whole / 1e6, 1),
                     "frac": round(STEP_BYTES_MASTER * N / ms_whole / 1e6 / peak, 4),
                     "launches": len(mp.mp_step_launches(0, N, opt.table))},
           "shards_8": {**LAST_TIMING, "ms": round(ms_sh, 5), "gparams_s": round(N / ms_sh / 1e6, 2),
                        "gbs": round(STEP_BYTES_MASTER * N / ms_sh / 1e6, 1),
                        "frac": round(STEP_BYTES_MASTER * N / ms_sh / 1e6 / peak, 4),
                        "launches": sum(len(mp.mp_step_launches(r * per, per, opt.table)) for r in range(8))},
           "what": "mp_adamw_step with fp32 master over the whole buffer vs 8 shard calls (global offsets r*N/8)"}
    del st, g, opt
    torch.cuda.empty_cache()
    return out


def measure_sr_stress(mp, stream, device, peak, n=64 << 20, steps=1000):
    """The stochastic-rounding stress set: 64M fp32 weights, |w| log-uniform
    in [1e-3, 10], random sign. (1) Throughput of the standalone rounding
    kernel on it (6 B per element). (2) A constant update of 1e-4 |w| per
    element (below half a bf16 step) for 1000 steps: the mean relative drift
    of the bf16 weights from the fp32 trajectory with stochastic rounding
    (mp_accumulate_sr: w = SR((float)w + delta), one kernel per step) and with
    round-to-nearest (the bf16 cast of (float)w + delta)."""
    w0 = W.sr_stress_weights(n, device=device)
    out16 = torch.empty(n, dtype=torch.bfloat16, device=device)
    ms = time_events(lambda: mp.mp_stochastic_round(out16, w0, 7, stream=stream), 20, stream)
    res = {"elements": n, "sr_kernel": {**LAST_TIMING, "ms": round(ms, 5), "gelems_s": round(n / ms / 1e6, 2),
                                        "gbs": round(SR_BYTES * n / ms / 1e6, 1),
                                        "frac": round(SR_BYTES * n / ms / 1e6 / peak, 4),
                                        "bytes_per_elem": SR_BYTES}}
    # the same launches back to back between one pair of events: each launch's
    # start overlaps the previous one's end (programmatic dependent launch),
    # so the per-launch latency that the figure above includes drops out; the
    # 403 MB per launch stay above the 129 MB L2, and every launch starts at
    # the front of the arrays, which the previous one left long ago
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    chained = 20
    a.record(stream)
    for _ in range(chained):
        mp.mp_stochastic_round(out16, w0, 7, stream=stream)
    b.record(stream)
    torch.cuda.synchronize()
    cms = a.elapsed_time(b) / chained
    res["sr_kernel_chained"] = {"ms": round(cms, 5), "launches": chained, "gelems_s": round(n / cms / 1e6, 2),
                                "gbs": round(SR_BYTES * n / cms / 1e6, 1),
                                "frac": round(SR_BYTES * n / cms / 1e6 / peak, 4),
                                "what": "mean over back-to-back launches between one pair of CUDA events"}
    delta = (w0.abs() * 1e-4).float()
    fp32 = w0.clone()
    sr = w0.to(torch.bfloat16)
    rne = w0.to(torch.bfloat16)
    tmp = torch.empty_like(w0)
    for t in range(1, steps + 1):
        fp32 += delta
        mp.mp_accumulate_sr(sr, delta, W.step_seed(t), stream=stream)
        torch.add(rne.float(), delta, out=tmp)
        rne.copy_(tmp)  # the round-to-nearest cast
    torch.cuda.synchronize()
    ref = fp32.double()
    res["drift"] = {"steps": steps, "update": "1e-4 |w0| per step",
                    "sr_mean_rel": float((sr.double() / ref - 1.0).mean()),
                    "rne_mean_rel": float((rne.double() / ref - 1.0).mean()),
                    "what": "mean over elements of bf16 weight / fp32 trajectory - 1 after the last step"}
    del w0, out16, delta, fp32, sr, rne, tmp
    torch.cuda.empty_cache()
    return res


def measure_e2e(mp, st, g, opt, N, stream, device, kw, iters, step_no):
    """Through the public API with host buffers: every step's bf16 gradients
    are copied from pinned host memory and the norm is read back to pinned
    host memory. Main figure: HostGradPipeline (the SMs copy step t's
    gradients, one block per SM, while the GPU updates step t - 1; one
    mp_optimizer_step call per step). Also reported: the same pipeline with a
    copy engine moving the gradients, and single mp_optimizer_step calls
    whose norm kernel reads the host gradients over the link itself (no
    overlap across steps)."""
    host_g = torch.empty(N, dtype=torch.bfloat16, pin_memory=True)
    host_g.copy_(g)
    host_norm = torch.empty(1, dtype=torch.float32, pin_memory=True)
    host_status = torch.empty(1, dtype=torch.int32, pin_memory=True)
    pipe = mp.HostGradPipeline(opt, device=device)

    def timed(step, n):
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            step()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    def pipelined():
        step_no[0] += 1
        t = step_no[0]
        pipe.step(st["params"], host_g, st["master"], st["m"], st["v"], t, W.step_seed(t), host_norm=host_norm,
                  stream=stream)
        host_status.copy_(opt.d_status, non_blocking=True)

    ms = timed(pipelined, iters)
    del pipe
    pipe = mp.HostGradPipeline(opt, device=device, transfer="engine")
    ms_engine = timed(pipelined, max(3, iters // 2))
    del pipe
    dev_g = torch.empty_like(g)

    def single_call():
        step_no[0] += 1
        t = step_no[0]
        opt.step(st["params"], dev_g, st["master"], st["m"], st["v"], t, W.step_seed(t), host_grads=host_g,
                 host_norm=host_norm, stream=stream)
        host_status.copy_(opt.d_status, non_blocking=True)

    ms_single = timed(single_call, max(3, iters // 2))
    return {"value": round(N * iters / (ms / 1e3) / 1e9, 3), "unit": UNIT, "h2d_bytes_per_step": 2 * N,
            "d2h_bytes_per_step": 8, "steps": iters, "ms_per_step": round(ms / iters, 5),
            "h2d": "bf16 grads from pinned host memory copied by the SMs (mp_copy_from_host, one block per SM) "
                   "beside the previous step's update",
            "api": "HostGradPipeline.step -> mp_copy_from_host + Optimizer.step (mp_optimizer_step)",
            "engine_copy": {"value": round(N * max(3, iters // 2) / (ms_engine / 1e3) / 1e9, 3),
                            "ms_per_step": round(ms_engine / max(3, iters // 2), 5),
                            "h2d": "the same pipeline with a copy engine (cudaMemcpyAsync) moving the gradients"},
            "single_call": {"value": round(N * max(3, iters // 2) / (ms_single / 1e3) / 1e9, 3),
                            "ms_per_step": round(ms_single / max(3, iters // 2), 5),
                            "h2d": "the norm kernel reads the pinned host gradients over the host link and "
                                   "writes the device copy (no overlap across steps)"}}


# ---------------------------------------------------------------------------
# CPU oracle (reported baseline; reference arm)
# ---------------------------------------------------------------------------
def prefix_entries(entries, n):
    out = []
    for e in entries:
        if e.offset >= n:
            break
        size = min(e.size, n - e.offset)
        out.append(W.Entry(W.TensorSpec(e.spec.name, (size,) if len(e.spec.shape) == 1 else (1, size),
                                        e.spec.kind), e.offset))
    return out


class OracleSample:
    """The first `n` params of the workload on the host, stepped by the oracle."""

    def __init__(self, n, workload=WORKLOAD):
        import oracle
        self.oracle = oracle
        entries = prefix_entries(W.layout(W.specs_for(workload)), n)
        self.tab = W.table(entries)
        st = W.make_state(workload, entries=entries)
        self.params = W.bf16_bits(st["params"]).copy()
        self.master = st["master"].numpy().copy()
        self.m = st["m"].numpy().copy()
        self.v = st["v"].numpy().copy()
        self.grads = [W.bf16_bits(W.make_grads(workload, s, entries=entries)).copy() for s in (1, 2)]
        self.n = n
        self.t = 0

    def step(self):
        H = W.HYPER
        self.t += 1
        g = self.grads[self.t % 2]
        _, _, scale = self.oracle.grad_norm(g, H["clip"])
        st = self.oracle.adamw_step(self.params, g, self.master, self.m, self.v, 0, self.tab, H["lr"], H["beta1"],
                                    H["beta2"], H["eps"], H["weight_decay"], float(scale), self.t,
                                    W.step_seed(self.t))
        assert st == 0


def host_cpu() -> dict:
    """The host's CPU model and core count, as the OS reports them."""
    model = platform.processor() or platform.machine()
    try:  # lscpu names Arm cores too (e.g. Neoverse-V2)
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        m = re.search(r"^Model name:\s*(.+)$", out, re.M)
        if m:
            return {"cpu_model": m.group(1).strip(), "nproc": os.cpu_count() or 1}
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            text = f.read()
        m = re.search(r"^model name\s*:\s*(.+)$", text, re.M)
        if m:
            model = m.group(1).strip()
        else:  # Arm hosts list an implementer and part number instead of a name
            impl = re.search(r"^CPU implementer\s*:\s*(\S+)", text, re.M)
            part = re.search(r"^CPU part\s*:\s*(\S+)", text, re.M)
            if impl and part:
                model = f"{platform.machine()} implementer {impl.group(1)} part {part.group(1)}"
    except OSError:
        pass
    return {"cpu_model": model, "nproc": os.cpu_count() or 1}


def cpu_baseline(seconds, workload=WORKLOAD):
    """The oracle on a prefix of the set: single-threaded (the reported
    value), and on every host core (`all_cores`)."""
    n = 1 << 22
    s = OracleSample(n, workload)
    s.step()
    t0 = time.perf_counter()
    steps = 0
    while time.perf_counter() - t0 < seconds:
        s.step()
        steps += 1
    dt = time.perf_counter() - t0
    out = {"value": round(n * steps / dt / 1e9, 5), "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": f"first {n} params of the {WORKLOAD_NAMES[workload]}, {steps} steps (norm + AdamW + SR), "
                     f"{dt:.1f} s, single-threaded C oracle", **host_cpu()}
    out["all_cores"] = cpu_baseline_all_cores(seconds, workload)
    return out


def cpu_baseline_all_cores(seconds, workload=WORKLOAD, n=1 << 24):
    """The same oracle on every host core: the norm as it stands (one thread,
    one sequential sum), then the step over contiguous shards, one thread
    each. Sharding the step changes no result (every element is independent
    given the scale), and the C calls release the GIL, so the shards run in
    parallel."""
    import threading
    cores = os.cpu_count() or 1
    s = OracleSample(n, workload)
    per = ((n + cores - 1) // cores + 7) // 8 * 8
    bounds = [(a, min(n, a + per)) for a in range(0, n, per)]
    H = W.HYPER

    def step():
        s.t += 1
        g = s.grads[s.t % 2]
        _, _, scale = s.oracle.grad_norm(g, H["clip"])
        status = []

        def shard(a, b):
            status.append(s.oracle.adamw_step(
                s.params[a:b], g[a:b], s.master[a:b], s.m[a:b], s.v[a:b], a, s.tab, H["lr"], H["beta1"],
                H["beta2"], H["eps"], H["weight_decay"], float(scale), s.t, W.step_seed(s.t)))
        threads = [threading.Thread(target=shard, args=ab) for ab in bounds]
        for th in threads:
            th.start()
        for th in threads:
            th.join()
        assert status == [0] * len(bounds)

    step()
    t0 = time.perf_counter()
    steps = 0
    while time.perf_counter() - t0 < seconds:
        step()
        steps += 1
    dt = time.perf_counter() - t0
    return {"value": round(n * steps / dt / 1e9, 5), "unit": UNIT, "cores": len(bounds), "kind": "oracle",
            "sample": f"first {n} params of the {WORKLOAD_NAMES[workload]}, {steps} steps, {dt:.1f} s: "
                      f"norm on one thread, "
                      f"step on {len(bounds)} threads over contiguous shards"}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    workload = args.workload
    budget = args.cpu_seconds if args.cpu_seconds else 30.0
    probe = OracleSample(1 << 18, workload)
    t0 = time.perf_counter()
    probe.step()
    per_param = (time.perf_counter() - t0) / probe.n
    total_steps = args.steps + args.warmup
    n = int(budget / max(1, total_steps) / per_param)
    n = max(1 << 12, min(n, 1 << 24)) & ~7
    s = OracleSample(n, workload)
    for _ in range(args.warmup):
        s.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        s.step()
    dt = time.perf_counter() - t0
    value = n * args.steps / dt / 1e9
    sample = (f"first {n} params of the {WORKLOAD_NAMES[workload]} per step (norm + AdamW + SR), "
              f"single-threaded C oracle")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD_NAMES[workload],
                       "params": W.total(W.layout(W.specs_for(workload))), "sample_params_per_step": n},
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample,
                             **host_cpu()},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU oracle sample budget")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_NAMES), default=WORKLOAD,
                    help="parameter set (default: the Llama-3-8B line)")
    ap.add_argument("--params", type=int, default=0,
                    help="use only the first P params of the set (small cases for profiling)")
    ap.add_argument("--kernel-samples", type=int, default=KERNEL_SAMPLES,
                    help="event-bracketed step calls after the timed region (at least 16)")
    ap.add_argument("--replicas", action="store_true",
                    help="with N > 1: an independent single-GPU step per rank instead of ZeRO-1")
    ap.add_argument("--zero1", action="store_true",
                    help="run the ZeRO-1 step even on one rank (a one-rank NCCL group)")
    ap.add_argument("--quick", action="store_true",
                    help="time the step only: no variants, end-to-end or CPU baseline")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    elif (world > 1 and not args.replicas) or args.zero1:
        line = run_zero1(args, world, rank, local)
    else:
        line = run_ours(args, world, rank, local)
    if torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()
    # anything a native library wrote to C stdio (e.g. NCCL's version line)
    # goes out before the JSON line, which stays the last line on stdout
    sys.stdout.flush()
    try:
        import ctypes
        ctypes.CDLL(None).fflush(None)
    except (OSError, AttributeError):
        pass
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
