"""Throughput of the fused attention forward on GB300.

One step = one attn_fwd call (the whole hot path: scheduling, TMA loads,
QK^T, softmax, correction, PV and the epilogue, plus the split-KV merge when
the workload splits) over the chosen workload, inputs resident in HBM.
Prints one JSON line on rank 0.

  python bench.py [--gpus N --steps K --warmup W] [--workload NAME] [--impl ours|reference]
                  [--schedule dynamic|static|grid] [--pair-cta auto|off|on] [--no-workloads]

After the headline workload (its JSON keys: value, roofline, e2e, clocks,
cpu_baseline), a one-GPU run also times every other workload the same way
(warm-up, K calls under CUDA events, clocks sampled) and reports each under
"workloads": kernel time, TFLOP/s and the fraction of the measured peak of
its own MMA types.

Multi-GPU (torchrun): every rank runs an independent replica of the workload
(weak scaling, no collective on the data path); value = FLOPs of all ranks /
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "mha_b4_h16_s4096_d128_causal"
METRIC = "attention fwd TFLOP/s at 1 GB300 and % of dense tensor peak (BF16/FP8)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_BYTES = 126 * 1024 * 1024
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "fa_tc05_d128_causal_b4h16s4096.md")


def kernel_source_hash():
    import glob
    import hashlib
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "attention_forward_sm100_gb300", "csrc", "*.cuh"))):
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, only while the
    kernel source still matches the one that was profiled."""
    if workload != DEFAULT_WORKLOAD or not os.path.exists(PROFILE_SUMMARY):
        return None
    fields = {}
    with open(PROFILE_SUMMARY) as f:
        for line in f:
            if ":" in line and not line.startswith("|"):
                k, _, v = line.partition(":")
                fields[k.strip()] = v.strip()
    if fields.get("kernel_source_sha256") != kernel_source_hash():
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--schedule", default="dynamic", choices=["dynamic", "static", "grid"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--pair-cta", default="auto", choices=["auto", "off", "on"],
                    help="CTA pairs for the headline workload")
    ap.add_argument("--no-workloads", action="store_true",
                    help="skip timing the other task workloads after the headline one")
    return ap.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def peak_tflops(spec, peaks, sustained=False):
    """Dense tensor peak for the workload's MMA mix (bf16 burst, or the
    sustained bf16 figure; FP8 runs at 2x the bf16 rate: all-FP8 at 2x, FP8
    QK^T with bf16 P.V blended as half the FLOPs at 2x)."""
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    bf16 = float(peaks.get(key, FALLBACK_PEAKS[key]))
    if spec.v_dtype == "fp8":
        return 2.0 * bf16
    if spec.qk_dtype == "fp8":
        return 2.0 / (1.0 / (2.0 * bf16) + 1.0 / bf16)
    return bf16


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.strip().split(",") for r in self.file.read().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower() in ("active", "1"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "window": "timed steps plus ~1 s of the same steps right after them"}


def cpu_baseline(spec, inputs, seconds):
    """The fp64 oracle timed on the host cores over whole (sequence, head)
    problems of the workload until `seconds` have passed; TFLOP/s of the
    visible pairs processed."""
    import numpy as np

    import oracle

    def f64(t):
        return None if t is None else t.float().double().numpy()

    cores = len(os.sched_getaffinity(0))
    lq, lk = spec.seq_lengths()
    from attention_forward_sm100_gb300.workloads import v_token_major
    q, k = f64(inputs["q"]), f64(inputs["k"])
    v = f64(v_token_major(inputs["v"], inputs.get("cu_seqlens_k"), inputs.get("cu_seqlens_v")))
    qr, kr = f64(inputs.get("q_rope")), f64(inputs.get("k_rope"))
    qs, ks = f64(inputs.get("q_scale")), f64(inputs.get("k_scale"))
    cu_q = inputs.get("cu_seqlens_q")
    cu_k = inputs.get("cu_seqlens_k")
    g = spec.heads_q // spec.heads_kv
    done_flops, heads = 0, 0
    t0 = time.perf_counter()
    order = [(b, h) for h in range(spec.heads_q) for b in range(spec.batch)]
    for b, h in order:
        hk = h // g
        if spec.varlen:
            a, e = int(cu_q[b]), int(cu_q[b + 1])
            c, f = int(cu_k[b]), int(cu_k[b + 1])
            args = (q[a:e, h], k[c:f, hk], v[c:f, hk], spec.softmax_scale, spec.causal,
                    None if qr is None else qr[a:e, h], None if kr is None else kr[c:f],
                    None if qs is None else qs[h, a:e], None if ks is None else ks[hk, c:f])
        else:
            args = (q[b, :, h], k[b, :, hk], v[b, :, hk], spec.softmax_scale, spec.causal,
                    None if qr is None else qr[b, :, h], None if kr is None else kr[b],
                    None if qs is None else qs[b, h], None if ks is None else ks[b, hk])
        oracle.attention_head(*args)
        n, m = lq[b], lk[b]
        pairs = (min(n, m) * (min(n, m) + 1) // 2 + max(0, n - m) * m) if spec.causal else n * m
        done_flops += 2 * (spec.d_qk + spec.rope + spec.d_v) * pairs
        heads += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    del np
    full = heads == spec.batch * spec.heads_q
    return {"value": done_flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{heads} whole (sequence, head) problems of {spec.batch * spec.heads_q}, "
                      f"fp64 numpy, {dt:.1f} s",
            "full_oracle_s": dt if full else dt * spec.flops() / done_flops,
            "full_oracle_s_kind": "measured" if full else "extrapolated (time per FLOP x all FLOPs)"}


def cpu_model():
    """Model name of the host CPU (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)   # this rank's GPU before any NCCL communicator exists
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank, world, ms):
    """Whole-job throughput: every rank ran flops_per_rank in at most ms."""
    return flops_per_rank * world / (ms * 1e-3) / 1e12


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# The task's workloads timed after the headline one in the same run (GPU
# only, no CPU leg): the small non-causal case, packed GQA, MLA with the
# shared rope part and FP8 Q/K; then the additions (all-FP8, split-KV, and
# split-KV of one long causal sequence with two heads); then the d128 and MLA
# workloads again on CTA pairs (label "+pairs").
OTHER_WORKLOADS = (("mha_b1_h2_s128_d64_noncausal", {}), ("varlen_gqa_b8_hq32_hkv8_d128_causal", {}),
                   ("mla_b2_h128_s4096_d128r64_causal", {}), ("fp8_b2_h32_s8192_d128_causal", {}),
                   ("fp8qkv_b2_h32_s8192_d128_causal", {}),
                   ("splitkv_b1_hq32_hkv8_sq256_sk32768_d128_noncausal", {}),
                   ("splitkv_b1_h2_s16384_d128_causal", {}),
                   ("mha_b4_h16_s4096_d128_causal", {"pair_cta": "on"}),
                   ("mla_b2_h128_s4096_d128r64_causal", {"pair_cta": "on"}))


def prepare(spec, dev, schedule):
    """Device inputs, outputs and the keyword arguments of pkg.forward for a
    workload; also the split count the library chose and kernels per call."""
    import torch

    import attention_forward_sm100_gb300 as pkg
    from attention_forward_sm100_gb300 import workloads as W
    inputs = W.make_inputs(spec)
    d = W.to_device(inputs, dev)
    lq, lk = spec.seq_lengths()
    out = torch.empty(d["q"].shape[:-1] + (spec.d_v,), dtype=torch.bfloat16, device=dev)
    if spec.varlen:
        lse = torch.empty((spec.heads_q, d["q"].shape[0]), dtype=torch.float32, device=dev)
    else:
        lse = torch.empty((spec.batch, spec.heads_q, spec.seqlen_q), dtype=torch.float32, device=dev)
    kw = dict(causal=spec.causal, softmax_scale=spec.softmax_scale, q_rope=d.get("q_rope"), k_rope=d.get("k_rope"),
              q_scale=d.get("q_scale"), k_scale=d.get("k_scale"), cu_seqlens_q=d.get("cu_seqlens_q"),
              cu_seqlens_k=d.get("cu_seqlens_k"), max_seqlen_q=max(lq), max_seqlen_k=max(lk), out=out, lse=lse,
              schedule=schedule, cu_seqlens_v=d.get("cu_seqlens_v"))
    prm = pkg.make_params(d["q"], d["k"], d["v"], **kw)
    ws = pkg.default_workspace(dev, pkg.workspace_bytes(prm))
    prm.workspace, prm.workspace_bytes = ws.data_ptr(), ws.numel()
    num_splits = pkg.plan(prm).num_splits
    return inputs, d, kw, out, lse, num_splits, (2 if num_splits > 1 else 1)


def time_calls(step, steps, stream):
    """Per-call device times (ms) of `steps` calls, CUDA events on `stream`.

    A short device-side sleep is queued ahead of the first event, so the first
    call is already enqueued when the GPU reaches it: the first interval then
    holds that call's device time and not the host's latency to issue it
    (the first event would otherwise be recorded on an idle GPU). Calls that
    take less device time than the host needs to issue one stay host-bound
    after the first."""
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    with torch.cuda.stream(stream):
        torch.cuda._sleep(200_000)          # ~0.1 ms at ~2 GHz: longer than one host call
    ev[0].record(stream)
    for i in range(steps):
        step()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)], ev[0].elapsed_time(ev[-1])


def soak(step, dev, seconds):
    """Keeps the same calls running so the clock sampler sees them."""
    import torch
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for _ in range(16):
            step()
        torch.cuda.synchronize(dev)


def small_call_latency(d, kw, stream, dev, calls=2000):
    """Per-call times of a problem small enough to be bound by the host path:
    back-to-back calls through ``forward`` (marshalling every call) and
    through a prepared call (``prepare``: one attn_fwd per call), wall time
    over `calls` calls; and the same call captured 100 times in a CUDA graph
    and replayed."""
    import torch

    import attention_forward_sm100_gb300 as pkg
    out = {}
    prep = pkg.prepare(d["q"], d["k"], d["v"], stream=stream, **kw)
    for name, fn in (("forward_us_per_call", lambda: pkg.forward(d["q"], d["k"], d["v"], stream=stream, **kw)),
                     ("prepared_us_per_call", prep.run)):
        for _ in range(50):
            fn()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(calls):
            fn()
        torch.cuda.synchronize(dev)
        out[name] = (time.perf_counter() - t0) * 1e6 / calls
    pkg.check(device=dev)
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream(dev)
    cs.wait_stream(stream)
    with torch.cuda.graph(g, stream=cs):
        for _ in range(100):
            pkg.forward(d["q"], d["k"], d["v"], stream=cs, **kw)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cs):          # replay() launches on the current stream
        g.replay()
        torch.cuda.synchronize(dev)
        g0.record(cs)
        for _ in range(5):
            g.replay()
        g1.record(cs)
    torch.cuda.synchronize(dev)
    out["graph_replay_us_per_call"] = g0.elapsed_time(g1) * 1e3 / 500
    pkg.check(device=dev)
    return out


def peak_label(spec, peak_src):
    if spec.v_dtype == "fp8":
        return f"2 x bf16 burst (fp8 Q/K/V), {peak_src}"
    if spec.qk_dtype == "fp8":
        return f"blended: half the FLOPs at 2 x bf16 burst (fp8 QK^T), half at bf16 burst, {peak_src}"
    return f"bf16 burst, {peak_src}"


def time_other_workloads(args, dev, stream, peaks, peak_src):
    """kernel_ms, TFLOP/s, fraction of the measured peak of the workload's
    own MMA types and clocks of every other workload, each timed like the
    headline one."""
    import torch

    import attention_forward_sm100_gb300 as pkg
    from attention_forward_sm100_gb300 import workloads as W
    res = {}
    for name, opts in OTHER_WORKLOADS:
        if name == args.workload and not opts:
            continue
        label = name + ("+pairs" if opts.get("pair_cta") == "on" else "")
        spec = W.WORKLOADS[name]
        inputs, d, kw, out, lse, splits, launches = prepare(spec, dev, args.schedule)
        kw = dict(kw, **opts)

        def step():
            pkg.forward(d["q"], d["k"], d["v"], stream=stream, **kw)

        for _ in range(max(3, args.warmup)):
            step()
        pkg.check(device=dev)
        clocks = ClockSampler(dev.index if dev.index is not None else 0)
        clocks.start()
        time.sleep(0.2)             # the sampler starts; the timed calls then run as a burst
        torch.cuda.synchronize(dev)
        for _ in range(max(3, args.warmup)):   # warm-up right before the timed calls (clocks up)
            step()
        per_call, _ = time_calls(step, args.steps, stream)
        soak(step, dev, 0.6)
        clk = clocks.stop()
        pkg.check(device=dev)
        kernel_ms = statistics.mean(per_call)
        flops = spec.flops()
        peak = peak_tflops(spec, peaks)
        achieved = flops / (kernel_ms * 1e-3) / 1e12
        entry = {"kernel_ms": kernel_ms, "median_ms": statistics.median(per_call), "tflops": achieved,
                 "frac": achieved / peak, "peak": peak, "peak_source": peak_label(spec, peak_src),
                 "flops_per_call": flops, "hbm_bytes_algorithmic": spec.hbm_bytes(), "num_splits": splits,
                 "gpu_launches": args.steps * launches, "steps": args.steps, "clocks": clk}
        if flops < 1e10:
            med = statistics.median(per_call)
            entry["us_per_call"] = med * 1e3
            entry["algorithmic_gbs"] = spec.hbm_bytes() / (med * 1e-3) / 1e9
            entry["latency"] = small_call_latency(d, kw, stream, dev)
        res[label] = entry
        del inputs, d, kw, out, lse
        torch.cuda.empty_cache()
    return res


def run_reference(args, spec, world, rank):
    """Reference arm: the CPU oracle as it stands, one bounded sample of the
    workload per step. Under torchrun only rank 0 runs and prints."""
    if rank != 0:
        return
    from attention_forward_sm100_gb300 import workloads as W
    inputs = W.make_inputs(spec)
    per_step = max(1.0, min(20.0, 100.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_baseline(spec, inputs, per_step / 4)
    vals = []
    last = None
    t0 = time.perf_counter()
    for _ in range(args.steps):
        last = cpu_baseline(spec, inputs, per_step)
        vals.append(last["value"])
    wall = time.perf_counter() - t0
    value = statistics.mean(vals)
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": wall * 1e3 / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": args.workload, "sample": last["sample"] if last else None},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": last["cores"], "kind": "oracle",
                             "sample": last["sample"]},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    from attention_forward_sm100_gb300 import workloads as W
    spec = W.WORKLOADS[args.workload]
    if args.impl == "reference":
        # No process group: the reference arm never communicates.
        run_reference(args, spec, int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")))
        return
    world, rank, local = dist_setup(args)

    import torch

    import attention_forward_sm100_gb300 as pkg
    if args.warmup < 3:
        args.warmup = 3
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    pkg.lib()
    stream = torch.cuda.current_stream(dev)
    # Kernels per call: the attention kernel, plus the merge kernel when the
    # library splits the keys of each query tile (split-KV).
    inputs, d, kw, out, lse, num_splits, launches_per_step = prepare(spec, dev, args.schedule)
    kw["pair_cta"] = args.pair_cta
    in_bytes = sum(t.numel() * t.element_size() for t in d.values() if isinstance(t, torch.Tensor))

    def step():
        pkg.forward(d["q"], d["k"], d["v"], stream=stream, **kw)

    for _ in range(args.warmup):
        step()
    pkg.check(device=dev)
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    time.sleep(0.3)                 # the sampler starts; the timed calls then run as a burst
    barrier(world)
    torch.cuda.synchronize(dev)
    for _ in range(args.warmup):    # the warm-up calls again, right before the timed ones (clocks up)
        step()
    per_launch, total_ms = time_calls(step, args.steps, stream)
    # The timed steps last milliseconds, nvidia-smi samples every 100 ms: keep
    # the same load running right after them until a second of samples exists.
    # These calls are timed too, in batches of 64, for the sustained figure:
    # the batches of the second half of that second run with the GPU at its
    # steady power and clock (the timed steps above are a burst from idle).
    t_soak = time.perf_counter()
    batches = []
    while time.perf_counter() - t_soak < 1.0:
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(64):
            step()
        b1.record(stream)
        torch.cuda.synchronize(dev)
        batches.append((time.perf_counter() - t_soak, b0.elapsed_time(b1) / 64))
    barrier(world)
    clk = clocks.stop()
    pkg.check(device=dev)
    median_ms = statistics.median(per_launch)
    # steady state: the batches that started after half of the second
    steady = [ms for t, ms in batches if t >= 0.5] or [ms for _, ms in batches]
    sus_ms = statistics.median(steady) if steady else None
    total_ms = max_over_ranks(total_ms, world, dev)
    ms = total_ms / args.steps
    flops = spec.flops()
    value = whole_job_tflops(flops, world, ms)
    kernel_ms = statistics.mean(per_launch)
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    peak = peak_tflops(spec, peaks)
    sustained = None
    if sus_ms:
        sus_peak = peak_tflops(spec, peaks, sustained=True)
        sus_value = flops / (sus_ms * 1e-3) / 1e12
        sustained = {"value": sus_value, "unit": "TFLOP/s", "ms_per_step": sus_ms, "peak": sus_peak,
                     "frac": sus_value / sus_peak, "batches": len(steady),
                     "peak_source": peak_label(spec, peak_src).replace("burst", "sustained"),
                     "window": "median of 64-call batches, each timed with CUDA events, that started in "
                               "the second half of the ~1 s of the same calls run after the timed steps"}

    # A problem this small is bound by the host's launch path: also time it
    # through a prepared call and replayed from a CUDA graph.
    small = small_call_latency(d, kw, stream, dev) if spec.flops() < 1e10 else None

    e2e = None
    if not args.no_e2e:
        # End to end through the public call with host buffers: every step
        # uploads its inputs from pinned host memory, runs the forward and
        # downloads O and LSE. Steps are pipelined the way a serving loop
        # would run them: two device buffer sets, the upload of step k+1 on
        # its own stream while step k computes and step k-1 downloads; the
        # timed region runs from the first upload to the last download.
        names = ("q", "k", "v", "q_rope", "k_rope", "q_scale", "k_scale", "cu_seqlens_q", "cu_seqlens_k",
                 "cu_seqlens_v")
        hin = {n: inputs[n].pin_memory() for n in names if inputs.get(n) is not None}
        h2d = sum(t.numel() * t.element_size() for t in hin.values())
        slots = []
        for b in range(2):
            din = {n: (d[n] if b == 0 else W.to_device({n: inputs[n]}, dev)[n]) for n in hin}
            o_b = out if b == 0 else torch.empty_like(out)
            l_b = lse if b == 0 else torch.empty_like(lse)
            ho = torch.empty(o_b.shape, dtype=o_b.dtype).pin_memory()
            hl = torch.empty(l_b.shape, dtype=l_b.dtype).pin_memory()
            slots.append(dict(din=din, o=o_b, lse=l_b, ho=ho, hl=hl,
                              loaded=torch.cuda.Event(), computed=torch.cuda.Event(), saved=torch.cuda.Event()))
        d2h = slots[0]["ho"].numel() * slots[0]["ho"].element_size() + \
            slots[0]["hl"].numel() * slots[0]["hl"].element_size()
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        kw_e = {k: v for k, v in kw.items() if k not in ("out", "lse") + names}

        def e2e_step(i):
            sl = slots[i % 2]
            up.wait_event(sl["computed"])              # the slot's previous forward has read its inputs
            with torch.cuda.stream(up):
                for n, t in hin.items():
                    sl["din"][n].copy_(t, non_blocking=True)
                sl["loaded"].record(up)
            stream.wait_event(sl["loaded"])
            stream.wait_event(sl["saved"])             # the slot's previous result has been downloaded
            di = sl["din"]
            pkg.forward(di["q"], di["k"], di["v"], q_rope=di.get("q_rope"), k_rope=di.get("k_rope"),
                        q_scale=di.get("q_scale"), k_scale=di.get("k_scale"), cu_seqlens_q=di.get("cu_seqlens_q"),
                        cu_seqlens_k=di.get("cu_seqlens_k"), cu_seqlens_v=di.get("cu_seqlens_v"), out=sl["o"],
                        lse=sl["lse"], stream=stream, **kw_e)
            sl["computed"].record(stream)
            down.wait_event(sl["computed"])
            with torch.cuda.stream(down):
                sl["ho"].copy_(sl["o"], non_blocking=True)
                sl["hl"].copy_(sl["lse"], non_blocking=True)
                sl["saved"].record(down)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n_e2e = max(4, min(args.steps, 12))
        e0.record(up)
        for i in range(n_e2e):
            e2e_step(i)
        e1.record(down)
        torch.cuda.synchronize(dev)
        pkg.check(device=dev)
        e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, world, dev)
        e2e = {"value": whole_job_tflops(flops, world, e_ms), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "pipelining": "2 buffer sets; upload, compute and download on their own streams"}

    cpu = None
    if rank == 0 and world >= 1 and not args.no_cpu_baseline and args.gpus == 1:
        cpu = cpu_baseline(spec, inputs, args.cpu_seconds)

    # The other workloads, after everything of the headline one (one GPU only).
    others = None
    if world == 1 and not args.no_workloads:
        del d, inputs
        others = time_other_workloads(args, dev, stream, peaks, peak_src)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": "fp8" if spec.v_dtype == "fp8" else ("fp8+bf16" if spec.qk_dtype == "fp8" else "bf16"),
            "data": "synthetic",
            "config": {"workload": args.workload, "batch": spec.batch, "heads_q": spec.heads_q,
                       "heads_kv": spec.heads_kv, "seqlen": spec.seqlen_q, "head_dim_qk": spec.d_qk + spec.rope,
                       "head_dim_v": spec.d_v, "causal": spec.causal, "flops_per_step": flops,
                       "seqlen_k": spec.seqlen_k, "num_splits": num_splits, "schedule": args.schedule,
                       "pair_cta": args.pair_cta,
                       "flops_tile_granular": spec.flops_tile_granular(),
                       "hbm_bytes_algorithmic": spec.hbm_bytes(),
                       "l2": "inputs larger than L2" if in_bytes > L2_BYTES else "inputs fit in L2 (no flush)",
                       "parallelism": f"replicas x{world}"},
            "pct_of_peak": 100.0 * value / world / peak,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak,
                         "peak_source": peak_label(spec, peak_src),
                         "traffic": profiled_traffic(args.workload) if args.pair_cta != "on" else None},
            "kernel_ms": kernel_ms,
            "median_ms": median_ms,
            "sustained": sustained,
            "clocks": clk,
            "gpu_launches": args.steps * launches_per_step,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "workloads": others,
        }
        if spec.qk_dtype == "fp8":
            # against the nominal dense peaks as well (FP8 4.5 PF, BF16 2.25 PF)
            line["pct_of_nominal"] = {"fp8_4500": 100.0 * value / world / 4500.0,
                                      "bf16_2250": 100.0 * value / world / 2250.0}
        if flops < 1e10:
            # a problem this small is bound by launch latency, not by the tensor cores
            hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
            line["latency"] = dict({"us_per_call": median_ms * 1e3,
                                    "algorithmic_gbs": spec.hbm_bytes() / (median_ms * 1e-3) / 1e9,
                                    "hbm_peak_gbs": hbm}, **small)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
