#!/usr/bin/env python
"""Benchmark of the GQA forward hot path on B300.

One step = one pass of the whole path over one batch of the non-causal
B=32, L=1024, h_q=8, g=4, d=64 workload (the pages' benchmark shape):
  1. kv_cache_append  the prompt's K/V (1024 tokens) into a [32, 4, 1025, 64] cache
  2. gqa_prefill_fwd  non-causal prefill, fp32 output
  3. kv_cache_append  one new token
  4. gqa_decode_fwd   one-token decode over the 1025 cached rows
value = algorithmic FLOPs of the step / device time of the step (TFLOP/s).
The dominant kernel (prefill) is also timed alone inside each step for the
roofline figure. After the timed region the script measures, for context,
the causal B=4 L=4096 h_q=32 g=8 d=128 prefill, the ragged B=64 decode over
a [64, 8, 8192, 128] cache and the B=16, S=32768 decode group-size sweep.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
Under torchrun each rank runs an independent replica on its own GPU.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GQA prefill TFLOP/s & decode KV-read GB/s vs roofline on 1×B300"
# DRAM bytes (read + write) of one prefill_kernel<64,false> launch of the bench workload, from
# the ncu capture summarised in profiles/prefill_noncausal_b32_l1024_hq8_g4_d64.md; reported
# only while prefill.cu is the source that was profiled (sha256 prefix below).
PROFILED_PREFILL = {"sha256_prefix": "041e011e5634ab7f", "dram_bytes": 67_179_008 + 20_607_232}
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
L2_FLUSH_BYTES = 256 << 20


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--no-extra", action="store_true", help="skip the context measurements")
    return p.parse_args(argv)


# --------------------------------------------------------------------- ranks

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(backend: str):
    import torch.distributed as dist

    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def reduce_max(x: float, device) -> float:
    """Max over ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, device) -> float:
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier():
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# --------------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """Samples SM clock and throttle reasons through NVML in a background thread."""

    REASONS = {
        0x0000000000000001: "gpu_idle",
        0x0000000000000002: "applications_clocks_setting",
        0x0000000000000004: "sw_power_cap",
        0x0000000000000008: "hw_slowdown",
        0x0000000000000020: "sync_boost",
        0x0000000000000040: "sw_thermal_slowdown",
        0x0000000000000080: "hw_thermal_slowdown",
        0x0000000000000100: "hw_power_brake_slowdown",
        0x0000000000000200: "display_clock_setting",
    }

    def __init__(self, device_index: int, period_s: float = 0.002):
        self.samples = []
        self.reasons = 0
        self.max_mhz = None
        self.error = None
        self._stop = threading.Event()
        self._period = period_s
        self._ok = False
        self._device_index = device_index
        try:
            import pynvml

            pynvml.nvmlInit()
            self._nv = pynvml
            self._h = pynvml.nvmlDeviceGetHandleByIndex(device_index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM)
            self._ok = True
        except Exception as e:  # fall back to the nvidia-smi CLI
            self.error = f"nvml: {type(e).__name__}: {e}"
            self._ok = False

    def _sample(self):
        nv = self._nv
        self.samples.append(nv.nvmlDeviceGetClockInfo(self._h, nv.NVML_CLOCK_SM))
        try:
            self.reasons |= nv.nvmlDeviceGetCurrentClocksEventReasons(self._h)
        except Exception:
            self.reasons |= nv.nvmlDeviceGetCurrentClocksThrottleReasons(self._h)

    def _smi_sample(self):
        import subprocess

        fields = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active")
        r = subprocess.run(["nvidia-smi", "-i", str(self._device_index),
                            f"--query-gpu={fields}", "--format=csv,noheader,nounits"],
                           capture_output=True, text=True, timeout=10)
        sm, mx, active = [x.strip() for x in r.stdout.strip().split(",")]
        self.samples.append(float(sm))
        self.max_mhz = float(mx)
        self.reasons |= int(active, 16)

    def _run(self):
        while not self._stop.is_set():
            try:
                self._sample() if self._ok else self._smi_sample()
            except Exception as e:
                self.error = (self.error or "") + f" sample: {e}"
                return
            time.sleep(self._period if self._ok else 0.05)

    def __enter__(self):
        try:
            self._sample() if self._ok else self._smi_sample()
        except Exception as e:
            self.error = (self.error or "") + f" first sample: {e}"
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        self._t.join()
        try:
            self._sample() if self._ok else self._smi_sample()
        except Exception:
            pass

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [],
                    "samples": 0, "error": self.error}
        reasons = [name for bit, name in self.REASONS.items() if self.reasons & bit]
        out = {"sm_mhz": float(statistics.median(self.samples)), "sm_max_mhz": self.max_mhz,
               "reasons": reasons, "samples": len(self.samples),
               "source": "nvml" if self._ok else "nvidia-smi"}
        if self.error:
            out["note"] = self.error
        return out


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info

        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


# --------------------------------------------------------------------- CPU oracle legs

def cpu_oracle_prefill_sample(budget_s: float, max_seqs: int = 32):
    """Time the fp64 oracle on whole sequences of the step's workload."""
    import numpy as np

    import oracle
    from grouped_query_attention_10_b300 import accounting, inputs

    w = inputs.NONCAUSAL_PREFILL
    q, k, v = inputs.prefill_inputs(w, device="cpu", B=max_seqs)
    f64 = lambda t: t.to(__import__("torch").float64).numpy()
    t0 = time.perf_counter()
    n = 0
    while n < max_seqs:
        oracle.prefill(f64(q[n:n + 1]), f64(k[n:n + 1]), f64(v[n:n + 1]), w.causal, w.scale)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    flops = accounting.prefill_flops(n, w.L, w.h_q, w.d, w.causal)
    del np
    return flops / dt / 1e12, n, dt


# --------------------------------------------------------------------- native arm

def native_arm(args):
    import torch

    from grouped_query_attention_10_b300 import accounting, inputs
    from grouped_query_attention_10_b300 import binding as gqa

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rank, world = dist_init("nccl")
    gqa.load_library()
    peaks, peak_src = load_peaks()

    w = inputs.NONCAUSAL_PREFILL
    B, L, h_q, g, d = w.B, w.L, w.h_q, w.g, w.d
    S_max = L + 1
    q, k, v = inputs.prefill_inputs(w, device=dev)
    k_new = inputs.random_bf16((B, 1, g, d), 2001, device=dev)
    v_new = inputs.random_bf16((B, 1, g, d), 2002, device=dev)
    q_new = inputs.random_bf16((B, h_q, d), 2003, device=dev)
    kc = torch.empty((B, g, S_max, d), dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    lens = torch.zeros((B,), dtype=torch.int32, device=dev)
    o = torch.empty((B, L, h_q, d), dtype=torch.float32, device=dev)
    od = torch.empty((B, h_q, d), dtype=torch.float32, device=dev)
    ws = torch.empty(gqa.gqa_decode_workspace_bytes(B, h_q, g, d, S_max), dtype=torch.uint8,
                     device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    from grouped_query_attention_10_b300.run_workload import make_l2_flush
    flush = make_l2_flush(dev)
    stream = torch.cuda.current_stream(dev)

    flops_prefill = accounting.prefill_flops(B, L, h_q, d, w.causal)
    flops_step = flops_prefill + accounting.decode_flops([S_max] * B, h_q, d)
    launches_per_step = 2 + 1 + 2 + 2  # append(rows, lens), prefill, append, decode(split, combine)

    def step_parts(s):
        # the step in three parts, split where the prefill is timed on its own
        def pre():
            lens.zero_()
            gqa.kv_cache_append(kc, vc, lens, k, v, status=status, stream=s)

        def pf():
            gqa.gqa_prefill_fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, status=status,
                                stream=s)

        def post():
            gqa.kv_cache_append(kc, vc, lens, k_new, v_new, status=status, stream=s)
            gqa.gqa_decode_fwd(q_new, kc, vc, lens, scale=w.scale, out=od, workspace=ws,
                               status=status, stream=s)
        return pre, pf, post

    eager_parts = step_parts(stream)

    def step():
        for fn in eager_parts:
            fn()

    for _ in range(max(args.warmup, 3)):
        flush()
        step()
    torch.cuda.synchronize()
    o_eager, od_eager = o.clone(), od.clone()

    # The timed steps replay the same library calls captured as CUDA graphs
    # (the launches of the small append / decode kernels then follow each
    # other without host round trips); the results must equal the eager ones.
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    graphs = []
    with torch.cuda.stream(cap):
        for fn in step_parts(cap):
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr, stream=cap):
                fn()
            graphs.append(gr)
    torch.cuda.synchronize()
    g_pre, g_pf, g_post = graphs

    def step_graph(ev_p0=None, ev_p1=None):
        g_pre.replay()
        if ev_p0 is not None:
            ev_p0.record(stream)
        g_pf.replay()
        if ev_p1 is not None:
            ev_p1.record(stream)
        g_post.replay()

    for _ in range(3):
        flush()
        step_graph()
    torch.cuda.synchronize()
    if not (torch.equal(o, o_eager) and torch.equal(od, od_eager)):
        raise RuntimeError("graph replay of the step differs from the eager calls")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            flush()  # L2 flush between timed steps, outside the timed interval
            e0, ep0, ep1, e1 = evs[i]
            e0.record(stream)
            step_graph(ep0, ep1)
            e1.record(stream)
        torch.cuda.synchronize()
    barrier()
    step_ms = [e[0].elapsed_time(e[3]) for e in evs]
    prefill_ms = [e[1].elapsed_time(e[2]) for e in evs]
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())} during the timed region")
    t_local = sum(step_ms) / 1e3
    t_max = reduce_max(t_local, dev)
    units = reduce_sum(flops_step * args.steps, dev)
    value = units / t_max / 1e12
    ms_per_step = t_max * 1e3 / args.steps

    import hashlib

    src = os.path.join(ROOT, "grouped_query_attention_10_b300", "csrc", "prefill.cu")
    with open(src, "rb") as f:
        same_kernel = hashlib.sha256(f.read()).hexdigest().startswith(
            PROFILED_PREFILL["sha256_prefix"])
    prefill_s = statistics.mean(prefill_ms) / 1e3
    achieved = flops_prefill / prefill_s / 1e12
    roofline = {"bound": "tensor", "kernel": "prefill_kernel<64,false>",
                "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                "peak_source": f"{peak_src} bf16 dense burst",
                "traffic": PROFILED_PREFILL["dram_bytes"] if same_kernel else None,
                "traffic_unit": "bytes per launch (ncu dram read+write)",
                "algorithmic_bytes": accounting.prefill_bytes(B, L, h_q, g, d, 4)}

    # ---- end to end: pinned host inputs in, results back, copies timed
    pin = lambda t: t.detach().to("cpu").pin_memory()
    h_in = [pin(x) for x in (q, k, v, k_new, v_new, q_new)]
    d_in = [q, k, v, k_new, v_new, q_new]
    h_o = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    h_od = torch.empty(od.shape, dtype=od.dtype, pin_memory=True)
    h2d = sum(x.numel() * x.element_size() for x in h_in)
    d2h = o.numel() * o.element_size() + od.numel() * od.element_size()

    def e2e_step():
        for hd, dd in zip(h_in, d_in):
            dd.copy_(hd, non_blocking=True)
        step()
        h_o.copy_(o, non_blocking=True)
        h_od.copy_(od, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2e_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    barrier()
    for a, b_ in e2e_evs:
        a.record(stream)
        e2e_step()
        b_.record(stream)
    torch.cuda.synchronize()
    e2e_t = reduce_max(sum(a.elapsed_time(b_) for a, b_ in e2e_evs) / 1e3, dev)
    e2e = {"value": round(units / e2e_t / 1e12, 3), "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": round(e2e_t * 1e3 / args.steps, 4)}

    result = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 3),
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "gqa_step_noncausal_b32_l1024_hq8_g4_d64",
                   "B": B, "L": L, "h_q": h_q, "g": g, "d": d, "causal": False,
                   "step": "append prompt K/V, prefill, append 1 token, decode 1 token",
                   "l2": "flushed between timed steps (256 MiB write, then 256 MiB read)",
                   "launch": "each step replays three CUDA graphs of the library calls "
                             "(reset + prompt append | prefill | token append + decode)",
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }

    if rank == 0 and world == 1:
        budget = float(os.environ.get("GQA_BENCH_CPU_BUDGET_S", "12"))
        tf, nseq, dt = cpu_oracle_prefill_sample(budget)
        result["cpu_baseline"] = {
            "value": tf, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"fp64 NumPy oracle prefill on {nseq} of the 32 sequences "
                      f"({dt:.1f} s); decode and append not included"}
    if not args.no_extra:
        result["extra"] = extra_measurements(dev, stream, peaks, peak_src)
    if rank == 0:
        print(json.dumps(result), flush=True)


def _time_calls(fn, n, stream, flush=None):
    import torch

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for a, b in evs:
        if flush is not None:
            flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) / 1e3 for a, b in evs]


def extra_measurements(dev, stream, peaks, peak_src):
    """Context measurements on the other workloads (not part of `value`)."""
    import torch

    from grouped_query_attention_10_b300 import accounting, inputs
    from grouped_query_attention_10_b300 import binding as gqa

    out = {}
    # causal Llama-style prefill; inputs + output exceed L2
    w = inputs.LLAMA_CAUSAL_PREFILL
    q, k, v = inputs.prefill_inputs(w, device=dev)
    o = torch.empty((w.B, w.L, w.h_q, w.d), dtype=torch.float32, device=dev)
    fn = lambda: gqa.gqa_prefill_fwd(q, k, v, causal=True, scale=w.scale, out=o, stream=stream)
    _time_calls(fn, 3, stream)
    ts = _time_calls(fn, 10, stream)
    flops = accounting.prefill_flops(w.B, w.L, w.h_q, w.d, True)
    tf = flops / statistics.median(ts) / 1e12
    out[w.name] = {"tflops": round(tf, 2), "ms": round(statistics.median(ts) * 1e3, 4),
                   "frac_of_bf16_peak": round(tf / peaks["bf16_tflops"], 4),
                   "peak_source": peak_src}
    del q, k, v, o
    torch.cuda.empty_cache()

    def decode_case(w):
        q, kc, vc, lens = inputs.decode_inputs(w, device=dev)
        o = torch.empty((w.B, w.h_q, w.d), dtype=torch.float32, device=dev)
        ws = torch.empty(gqa.gqa_decode_workspace_bytes(w.B, w.h_q, w.g, w.d, w.S_max),
                         dtype=torch.uint8, device=dev)
        from grouped_query_attention_10_b300.run_workload import make_l2_flush
        flush = make_l2_flush(dev)
        fn = lambda: gqa.gqa_decode_fwd(q, kc, vc, lens, scale=w.scale, out=o, workspace=ws,
                                        stream=stream)
        _time_calls(fn, 3, stream, flush)
        ts = _time_calls(fn, 10, stream, flush)
        nbytes = accounting.decode_kv_bytes(lens.tolist(), w.g, w.d)
        t = statistics.median(ts)
        gbs = nbytes / t / 1e9
        return {"gbs": round(gbs, 1), "us": round(t * 1e6, 2), "kv_bytes": nbytes,
                "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4), "peak_source": peak_src}

    out[inputs.DECODE_RAGGED.name] = decode_case(inputs.DECODE_RAGGED)
    torch.cuda.empty_cache()
    sweep = {}
    for g in inputs.DECODE_SWEEP_G:
        sweep[f"g{g}"] = decode_case(inputs.decode_sweep(g))
        torch.cuda.empty_cache()
    out["decode_sweep_b16_hq32_d128_s32768"] = sweep
    return out


# --------------------------------------------------------------------- reference arm

def reference_arm(args):
    """The CPU oracle, timed as it stands, on bounded samples of the workload."""
    import torch

    import oracle
    from grouped_query_attention_10_b300 import accounting, inputs

    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = inputs.NONCAUSAL_PREFILL
    n_seq = 4
    q, k, v = inputs.prefill_inputs(w, device="cpu", B=n_seq)
    f64 = lambda t: t.to(torch.float64).numpy()
    qs, ks, vs = f64(q), f64(k), f64(v)

    def step(i):
        b = i % n_seq
        oracle.prefill(qs[b:b + 1], ks[b:b + 1], vs[b:b + 1], w.causal, w.scale)

    for i in range(max(args.warmup, 1)):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    flops = accounting.prefill_flops(1, w.L, w.h_q, w.d, w.causal) * args.steps
    value = flops / dt / 1e12
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": max(args.warmup, 1),
        "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "gqa_step_noncausal_b32_l1024_hq8_g4_d64", "B": w.B, "L": w.L,
                   "h_q": w.h_q, "g": w.g, "d": w.d, "causal": False,
                   "parallelism": "cpu, rank 0 only"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(),
                         "kind": "oracle",
                         "sample": "fp64 NumPy oracle prefill of one sequence "
                                   "(8 heads x 1024 x 1024) per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        reference_arm(args)
    else:
        native_arm(args)


if __name__ == "__main__":
    main()
