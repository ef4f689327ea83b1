#!/usr/bin/env python
"""Benchmark of the attention hot path on GB300.

One step = one attention forward on the non-causal prefill workload
(B8 Hq32 Hkv32 Nq=Nk=8192 D128, bf16) followed by one split-KV decode on the
decode workload (B8 Hq32 Hkv8 Nk65536 D128, nsplit 32).  Inputs are seeded
synthetic bf16 tensors resident in HBM; each input tensor is larger than the
129 MB L2, so no flush is needed between steps.

Headline: prefill bf16 TFLOP/s = 4*B*Hq*Nq*Nk*D / (prefill kernel time);
the decode line reports algorithmic HBM GB/s (K/V cache once + q + o + lse)
over split + combine time.  Rank 0 prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun (N > 1) every rank runs the same per-GPU work on its own GPU
(weak scaling, no collective on the data path); the timing is the max over
ranks.  ``--impl reference`` times the CPU fp64 oracle (the only reference
this path has) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "attn fwd bf16 TFLOPS vs 2.25 PF peak; split-KV decode HBM GB/s"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-other", action="store_true",
                    help="skip timing the other prefill workloads (causal, long GQA, tiny)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    return args


# ----------------------------------------------------------------------------- ranks


def dist_setup(backend):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value across ranks (the slowest rank sets the job time)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- helpers


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, \
            "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_HEADERS = ("ptx.cuh", "internal.h")  # included by every kernel file


def kernel_source_hash(name: str) -> str:
    """sha256 (first 16 hex digits) of a kernel source file and the headers
    it includes: a profile taken before any of them changed is stale."""
    h = hashlib.sha256()
    for f in (name, *KERNEL_HEADERS):
        with open(os.path.join(ROOT, "attention_forward_sm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_file: str, key: str):
    """dram read+write bytes per launch from the committed ncu summary, or None
    when there is none or the kernel source changed since it was captured."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)[key]
    except (OSError, KeyError, ValueError):
        return None
    if d.get("source_sha256_16") != kernel_source_hash(kernel_file):
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None, "samples": len(rows),
                "reasons": reasons}


# ----------------------------------------------------------------------------- oracle timing


def time_oracle(w, q_h, k_h, v_h, nrows, seed=3):
    """Time the CPU fp64 oracle on `nrows` sampled query rows of workload w.
    Returns (seconds, flops of the sample, threads used, description)."""
    import oracle
    from attention_forward_sm_gb300 import workloads as W
    rows = W.sample_rows(w, nrows, seed=seed).numpy()[:nrows]
    if w.causal:
        keys = sum(min(int(r) % w.Nq + 1, w.Nk) for r in rows)
    else:
        keys = len(rows) * w.Nk
    flops = 4.0 * keys * w.D
    nthreads = os.cpu_count() or 1
    lib = oracle.load()
    t0 = time.perf_counter()
    oracle.attn_rows(q_h, k_h, v_h, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.D, w.causal, w.scale, rows,
                     nthreads=nthreads, lib=lib)
    dt = time.perf_counter() - t0
    return dt, flops, nthreads, f"{len(rows)} sampled query rows of {w.label()}"


# ----------------------------------------------------------------------------- reference arm


def run_reference(args):
    rank, world = dist_setup("gloo")
    if rank != 0:
        return 0
    import torch
    from attention_forward_sm_gb300 import workloads as W
    w = W.WORKLOADS["prefill"]
    q, k, v = W.make_inputs(w, "cpu")
    total = args.steps + args.warmup
    per_step = max(16, min(1024, 8192 // total))
    for _ in range(args.warmup):
        time_oracle(w, q, k, v, per_step, seed=1)
    secs, flops = 0.0, 0.0
    threads, desc = 1, ""
    for i in range(args.steps):
        dt, fl, threads, desc = time_oracle(w, q, k, v, per_step, seed=100 + i)
        secs += dt
        flops += fl
    value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.label(), "global_batch": w.B, "seq_len": w.Nq,
                   "sample_per_step": f"{per_step} query rows"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{per_step} rows per step; {desc}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    del torch
    return 0


# ----------------------------------------------------------------------------- GPU arm


def run_gpu(args):
    import torch
    rank, world = dist_setup("nccl")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from attention_forward_sm_gb300 import _build
    from attention_forward_sm_gb300 import binding as attn
    from attention_forward_sm_gb300 import workloads as W
    if rank == 0 or world == 1:
        _build.build()
    barrier(world)
    attn.load()

    wp, wd = W.WORKLOADS["prefill"], W.WORKLOADS["decode"]
    q, k, v = W.make_inputs(wp, dev)
    o = torch.empty_like(q)
    lse = torch.empty((wp.B, wp.Hq, wp.Nq), dtype=torch.float32, device=dev)
    dq, dk, dv = W.make_inputs(wd, dev)
    do = torch.empty_like(dq)
    dlse = torch.empty((wd.B, wd.Hq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def prefill():
        attn.attn_fwd(q, k, v, o, lse, wp.B, wp.Hq, wp.Hkv, wp.Nq, wp.Nk, wp.D, wp.causal,
                      wp.scale, sh)

    def decode():
        attn.attn_decode_splitkv(dq, dk, dv, do, dlse, wd.B, wd.Hq, wd.Hkv, wd.Nk, wd.D,
                                 wd.nsplit, sh)

    for _ in range(args.warmup):
        prefill()
        decode()
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize(dev)
        start.record(stream)
        for i in range(K):
            ev[i][0].record(stream)
            prefill()
            ev[i][1].record(stream)
            decode()
            ev[i][2].record(stream)
        end.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    clocks = clk.summary()
    total_ms = max_over_ranks(start.elapsed_time(end), world, dev)
    pf_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    dec_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    pf_sum = max_over_ranks(sum(pf_ms), world, dev)
    dec_sum = max_over_ranks(sum(dec_ms), world, dev)
    if attn.attn_get_device_error(sh) != 0:
        raise RuntimeError("a kernel reported a timed-out wait during the benchmark")

    flops = wp.flops()
    tflops = world * K * flops / (pf_sum * 1e-3) / 1e12
    dec_gbs = world * K * wd.decode_bytes() / (dec_sum * 1e-3) / 1e9
    peaks, peak_kind = load_peaks()
    pf_avg_s = statistics.mean(pf_ms) * 1e-3
    dec_avg_s = statistics.mean(dec_ms) * 1e-3
    achieved = flops / pf_avg_s / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "traffic": profiled_traffic("fwd_sm103a.cu", "attn_fwd_kernel"),
                "peak_kind": f"{peak_kind} bf16 dense, burst (kernel timed in a sub-second loop)",
                "kernel": "attn_fwd_kernel<128>", "flops_per_launch": flops,
                "frac_of_nominal_2250": achieved / 2250.0}
    dec_achieved = wd.decode_bytes() / dec_avg_s / 1e9
    decode_line = {
        "workload": wd.label(), "value": dec_gbs, "unit": "GB/s", "ms_per_call": 1e3 * dec_avg_s,
        "roofline": {"bound": "hbm", "achieved": dec_achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": dec_achieved / peaks["hbm_gbs"],
                     "traffic": profiled_traffic("decode_sm103a.cu", "decode_split_kernel"),
                     "peak_kind": f"{peak_kind} copy bandwidth",
                     "bytes_per_call": wd.decode_bytes(),
                     "kernels": "decode_split_kernel<128,4> + decode_combine_kernel<128>"},
    }

    other = dec_graph = None
    if not args.no_other:
        other = time_other_workloads(attn, W, dev, peaks["bf16_tflops"])
        dec_graph = time_decode_graph(attn, W, dev, wd)
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, attn, W, wp, wd, dev, world)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        q_h, k_h, v_h = q.cpu(), k.cpu(), v.cpu()
        dt, fl, threads, desc = time_oracle(wp, q_h, k_h, v_h, 32768)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": desc, "seconds": dt,
               # the whole workload at the sample's rate (every row costs the same)
               "extrapolated_full_workload_seconds": dt * wp.flops() / fl}

    line = {
        "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wp.label(), "global_batch": wp.B * world, "seq_len": wp.Nq,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "decode_workload": wd.label(),
                   "l2": "inputs larger than L2 (each q/k/v tensor >= 537 MB), no flush"},
        "roofline": roofline,
        "decode": decode_line,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": 3 * K,
        "clocks": clocks,
        "prefill_ms_per_call": 1e3 * pf_avg_s,
        # spread of the per-call prefill times over the timed steps (clock and
        # power behaviour under sustained load shows here)
        "prefill_ms_per_call_stats": {"min": min(pf_ms), "median": statistics.median(pf_ms),
                                      "max": max(pf_ms),
                                      "first_quarter_mean": statistics.mean(pf_ms[:max(1, K // 4)]),
                                      "last_quarter_mean": statistics.mean(pf_ms[-max(1, K // 4):])},
        "other_prefill_workloads": other,
        "decode_graph": dec_graph,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def time_other_workloads(attn, W, dev, peak_tflops, calls=3, rest_s=1.0):
    """CUDA-event time of the other prefill workloads (separate from the step):
    returns {name: {...}} with TFLOP/s (causal flops halved).  Each timed
    region starts after `rest_s` seconds of idle GPU, so that a workload does
    not inherit the clock state the timed step loop (or the workload before
    it) left behind: right after the step loop the D = 64 workload measures
    ~7-10 % lower than on a rested GPU, which it matches again after ~1 s."""
    import time
    import torch
    out = {}
    d64 = W.custom(8, 32, 32, 8192, 8192, 64, False, seed_index=960)
    for name in ("causal", "long_gqa", "tiny", "d64"):
        w = d64 if name == "d64" else W.WORKLOADS[name]
        q, k, v = W.make_inputs(w, dev)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
        stream = torch.cuda.current_stream(dev)

        def call():
            attn.attn_fwd(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.D, w.causal, w.scale,
                          stream.cuda_stream)

        n = calls if name != "tiny" else 50
        for _ in range(3):
            call()
        torch.cuda.synchronize(dev)
        time.sleep(rest_s)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            call()
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms = a.elapsed_time(b) / n
        tf = w.flops() / (ms * 1e-3) / 1e12
        out[name] = {"workload": w.label(), "ms_per_call": ms, "tflops": tf,
                     "frac_of_measured_peak": tf / peak_tflops, "frac_of_nominal_2250": tf / 2250.0,
                     "calls": n, "idle_s_before_timing": rest_s}
        del q, k, v, o, lse
        torch.cuda.empty_cache()
    # FP8 (E4M3) inputs on the prefill shapes: same flop count, the peak is the
    # measured bf16 one times the nominal fp8 / bf16 ratio (2)
    for name in ("prefill", "causal"):
        w = W.WORKLOADS[name]
        q8, k8, _, vt8 = W.make_inputs_fp8(w, dev)
        o = torch.empty((w.B, w.Hq, w.Nq, w.D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
        stream = torch.cuda.current_stream(dev)
        sc = W.FP8_SCALES

        def call():
            attn.attn_fwd_fp8(q8, k8, vt8, o, lse, w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.D, w.causal,
                              w.scale, sc["q"], sc["k"], sc["v"], stream.cuda_stream)

        for _ in range(3):
            call()
        torch.cuda.synchronize(dev)
        time.sleep(rest_s)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(calls):
            call()
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms = a.elapsed_time(b) / calls
        tf = w.flops() / (ms * 1e-3) / 1e12
        out[f"fp8_{name}"] = {"workload": "e4m3 " + w.label(), "ms_per_call": ms, "tflops": tf,
                              "frac_of_fp8_peak": tf / (2.0 * peak_tflops),
                              "fp8_peak": 2.0 * peak_tflops,
                              "fp8_peak_kind": "measured bf16 burst x 2 (nominal fp8/bf16 ratio)",
                              "frac_of_nominal_4500": tf / 4500.0, "calls": calls,
                              "idle_s_before_timing": rest_s}
        del q8, k8, vt8, o, lse
        torch.cuda.empty_cache()
    return out


def time_decode_graph(attn, W, dev, wd, calls=200):
    """Decode step as a replayed CUDA graph vs the direct call, on the decode
    workload and on a short-context step (B1 Hq32 Hkv8 Nk4096) where fixed
    costs weigh most.  Per call: GPU time between CUDA events over `calls`
    back-to-back calls, and the host time to enqueue them."""
    import torch
    out = {}
    small = W.custom(1, 32, 8, 1, 4096, 128, False, seed_index=950, decode=True, nsplit=8)
    for name, w, n in (("decode", wd, 20), ("short_context", small, calls)):
        q, k, v = W.make_inputs(w, dev)
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.Hq), dtype=torch.float32, device=dev)
        stream = torch.cuda.current_stream(dev)
        sh = stream.cuda_stream
        g = attn.DecodeGraph(q, k, v, w.nsplit)

        def direct():
            attn.attn_decode_splitkv(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.Nk, w.D, w.nsplit, sh)

        def noalloc():
            attn.attn_decode_splitkv_noalloc(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.Nk, w.D,
                                             w.nsplit, sh)

        def graph():
            attn.attn_decode_graph_launch(g.handle, sh)

        res = {"workload": w.label(), "calls": n}
        for label, fn in (("direct", direct), ("noalloc", noalloc), ("graph", graph)):
            for _ in range(5):
                fn()
            torch.cuda.synchronize(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            t0 = time.perf_counter()
            for _ in range(n):
                fn()
            host_s = time.perf_counter() - t0
            b.record(stream)
            torch.cuda.synchronize(dev)
            res[f"{label}_us_per_call"] = 1e3 * a.elapsed_time(b) / n
            res[f"{label}_host_enqueue_us_per_call"] = 1e6 * host_s / n
        torch.cuda.synchronize(dev)
        if not (torch.equal(o, g.o) and torch.equal(lse, g.lse)):
            raise RuntimeError("graph replay and direct decode differ")
        res["graph_gbs"] = w.decode_bytes() / (res["graph_us_per_call"] * 1e-6) / 1e9
        g.close()
        out[name] = res
        del q, k, v, o, lse
        torch.cuda.empty_cache()
    return out


def run_e2e(args, attn, W, wp, wd, dev, world):
    """Same step through the C ABI with host buffers: pinned H2D copies of the
    step's inputs, the two calls, D2H of the results, all inside the timed
    region."""
    import torch
    pin = dict(device="cpu", pin_memory=True)
    hq, hk, hv = W.make_inputs(wp, dev)
    host_in = [t.to("cpu").pin_memory() for t in (hq, hk, hv)]
    dhq, dhk, dhv = W.make_inputs(wd, dev)
    host_din = [t.to("cpu").pin_memory() for t in (dhq, dhk, dhv)]
    del hq, hk, hv, dhq, dhk, dhv
    dev_din = [torch.empty_like(t, device=dev) for t in host_din]
    do = torch.empty_like(dev_din[0])
    dlse = torch.empty((wd.B, wd.Hq), dtype=torch.float32, device=dev)
    h_o = torch.empty(host_in[0].shape, dtype=host_in[0].dtype, **pin)
    h_lse = torch.empty((wp.B, wp.Hq, wp.Nq), dtype=torch.float32, **pin)
    h_do = torch.empty(do.shape, dtype=do.dtype, **pin)
    h_dlse = torch.empty(dlse.shape, dtype=dlse.dtype, **pin)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def step(record=None):
        # prefill: host buffers in and out through attn_fwd_host, whose copies
        # in, compute and copies out overlap unit by unit
        attn.attn_fwd_host(host_in[0], host_in[1], host_in[2], h_o, h_lse, wp.B, wp.Hq, wp.Hkv,
                           wp.Nq, wp.Nk, wp.D, wp.causal, wp.scale, sh)
        if record is not None:
            record.record(stream)
        for d, h in zip(dev_din, host_din):
            d.copy_(h, non_blocking=True)
        attn.attn_decode_splitkv(dev_din[0], dev_din[1], dev_din[2], do, dlse, wd.B, wd.Hq,
                                 wd.Hkv, wd.Nk, wd.D, wd.nsplit, sh)
        h_do.copy_(do, non_blocking=True)
        h_dlse.copy_(dlse, non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    K = max(1, args.e2e_steps)
    marks = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
              torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize(dev)
    for i in range(K):
        marks[i][0].record(stream)
        step(record=marks[i][1])
        marks[i][2].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    pf = max_over_ranks(sum(m[0].elapsed_time(m[1]) for m in marks), world, dev)
    dec = max_over_ranks(sum(m[1].elapsed_time(m[2]) for m in marks), world, dev)
    h2d = sum(t.numel() * t.element_size() for t in host_in + host_din)
    d2h = sum(t.numel() * t.element_size() for t in (h_o, h_lse, h_do, h_dlse))
    return {"value": world * K * wp.flops() / (pf * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": (pf + dec) / K,
            "decode_gbs": world * K * wd.decode_bytes() / (dec * 1e-3) / 1e9,
            "steps": K, "path": "prefill: attn_fwd_host on pinned host buffers (copies in, "
                                "compute and copies out pipelined per (batch, KV-head block)); "
                                "decode: pinned host -> device copies, attn_decode_splitkv, "
                                "device -> pinned host copies (C ABI via ctypes)"}


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
