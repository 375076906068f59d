#!/usr/bin/env python
"""Benchmark of the GQA forward hot path on B300.

One step = one pass of the whole path over one batch of the Llama-style causal
workload B=4, L=4096, h_q=32, g=8, d=128:
  1. kv_cache_append  the prompt's K/V (4096 tokens) into a [4, 8, 4097, 128] cache
  2. gqa_prefill_fwd  causal prefill, bf16 output (fp32 accumulation)
  3. kv_cache_append  one new token
  4. gqa_decode_fwd   one-token decode over the 4097 cached rows
value = algorithmic FLOPs of the step (causal pairs only) / device time of the
step (TFLOP/s). The dominant kernel (the prefill) is also timed alone inside
each step for the roofline figure.

The decode half of the metric is measured on the ragged decode workload
(B=64, h_q=32, g=8, d=128, cache [64, 8, 8192, 128], lengths uniform in
[1024, 8192]); its KV-read rate and roofline go in ``roofline["decode"]``.
After that the script measures, for context (``extra``), the pages' non-causal
benchmark shape B=32 L=1024 h_q=8 g=4 d=64, the B=16 S=32768 decode group-size
sweep and the variant workloads (sliding window, ALiBi, chunked prefill,
paged decode, windowed decode, prompt appends).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
Under torchrun each rank runs an independent replica on its own GPU.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GQA prefill TFLOP/s & decode KV-read GB/s vs roofline on 1×B300"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# Vendor figures, reported beside the measured peaks: dense bf16 tensor rate
# and HBM3e bandwidth of one B300.
NOMINAL_BF16_TFLOPS = 2250.0
NOMINAL_HBM_GBS = 8000.0
# The step's outputs are stored in the input dtype (bf16); every product,
# the softmax and the accumulation run in fp32.
OUT_DTYPE_NAME = "bf16"
# DRAM bytes (read + write) per launch from the committed ncu captures of the
# two roofline kernels, valid only while the kernel sources hash to the
# prefix given (sha256 over the listed files, concatenated in order).
PROFILED = {
    # ncu --set full of one prefill_kernel<128,causal> launch of the causal workload
    # (output dtype as given: the traffic counts the output writes)
    "prefill_causal_d128": {"files": ["prefill.cu", "ptx.cuh"], "out": "bf16",
                            "sha256_prefix": "3e2c4bf7f9b14d7f",
                            "dram_bytes": 312_190_464 + 79_479_552},
    # ncu --set full of one decode_split_kernel<128,1> launch of the B=64 ragged decode
    "decode_ragged": {"files": ["decode.cu", "ptx.cuh"], "sha256_prefix": "17cd1b6cc220a6ec",
                      "dram_bytes": 1_139_230_000 + 12_160_512},
}


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--no-extra", action="store_true", help="skip the context measurements")
    p.add_argument("--step-only", action="store_true",
                   help="time the step and print its line without the decode roofline, e2e, "
                        "CPU and context legs (for launch lists under a profiler)")
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


def source_sha(files) -> str:
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(ROOT, "grouped_query_attention_10_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(key: str, out: str = None):
    """ncu DRAM bytes per launch of a roofline kernel, or None when the kernel
    source has changed since the capture (or the capture wrote another output
    dtype than the one asked for)."""
    p = PROFILED[key]
    if not p["sha256_prefix"] or p["dram_bytes"] is None:
        return None
    if out is not None and p.get("out") != out:
        return None
    return p["dram_bytes"] if source_sha(p["files"]).startswith(p["sha256_prefix"]) else None


class ClockSampler:
    """Samples the SM clock and the clock-event reasons with `nvidia-smi -lms`
    in a child process while the timed region runs."""

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
    FIELDS = "clocks.sm,clocks.max.sm,clocks_event_reasons.active"

    def __init__(self, device_index: int, period_ms: int = 50):
        self.device = str(device_index)
        try:
            import torch

            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            if uuid:
                self.device = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        self.period_ms = period_ms
        self.proc = None
        self.lines = []
        self.error = None

    def _query_once(self):
        r = subprocess.run(["nvidia-smi", "-i", self.device, f"--query-gpu={self.FIELDS}",
                            "--format=csv,noheader,nounits"], capture_output=True, text=True,
                           timeout=20)
        return r.stdout.strip().splitlines()

    def __enter__(self):
        try:
            self.lines += self._query_once()
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.device, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._reader = threading.Thread(target=self._read, daemon=True)
            self._reader.start()
        except Exception as e:
            self.error = f"nvidia-smi: {type(e).__name__}: {e}"
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=10)
            except Exception:
                self.proc.kill()
            self._reader.join(timeout=5)
        try:
            self.lines += self._query_once()
        except Exception:
            pass

    def summary(self):
        sm, mx, reasons = [], None, 0
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) != 3:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
                reasons |= int(parts[2], 16)
            except ValueError:
                continue
        out = {"sm_mhz": float(statistics.median(sm)) if sm else None, "sm_max_mhz": mx,
               "reasons": [n for bit, n in self.REASONS.items() if reasons & bit],
               "samples": len(sm), "source": f"nvidia-smi -lms {self.period_ms}"}
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


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def _time_calls(fn, n, stream, flush=None):
    """CUDA-event time of n calls of fn on `stream` (seconds each); the L2
    flush, when given, runs before every call, outside the timed interval."""
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


# --------------------------------------------------------------------- CPU oracle legs

def _group_slice(q, k, v, b, kvh, G):
    """Sequence b, K/V head kvh and its G query heads, as fp64 arrays."""
    import torch

    f64 = lambda t: t.to(torch.float64).numpy()
    return (f64(q[b:b + 1, :, kvh * G:(kvh + 1) * G]), f64(k[b:b + 1, :, kvh:kvh + 1]),
            f64(v[b:b + 1, :, kvh:kvh + 1]))


def oracle_prefill_block(qs, ks, vs, r0, rows, scale):
    """The oracle on query rows [r0, r0 + rows) of one causal K/V group over
    keys [0, r0 + rows); returns the FLOPs that block represents."""
    import oracle

    r1 = min(r0 + rows, qs.shape[1])
    oracle.prefill(qs[:, r0:r1], ks[:, :r1], vs[:, :r1], True, scale, q_offset=r0)
    pairs = sum(i + 1 for i in range(r0, r1))
    return 4 * qs.shape[2] * qs.shape[3] * pairs


def cpu_oracle_prefill_sample(budget_s: float, rows: int = 512):
    """Time the fp64 oracle on whole K/V groups of the causal workload, in
    blocks of query rows, until the time budget is spent."""
    from grouped_query_attention_10_b300 import inputs

    w = inputs.LLAMA_CAUSAL_PREFILL
    q, k, v = inputs.prefill_inputs(w, device="cpu", B=1)
    G = w.h_q // w.g
    flops, groups, t0 = 0, 0, time.perf_counter()
    for kvh in range(w.g):
        qs, ks, vs = _group_slice(q, k, v, 0, kvh, G)
        for r0 in range(0, w.L, rows):
            flops += oracle_prefill_block(qs, ks, vs, r0, rows, w.scale)
        groups += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, groups, dt


def cpu_oracle_decode_sample(budget_s: float, max_seqs: int = 64):
    """Time the fp64 oracle decode on whole sequences of the ragged workload."""
    import torch

    import oracle
    from grouped_query_attention_10_b300 import accounting, inputs

    w = inputs.DECODE_RAGGED
    q, kc, vc, lens = inputs.decode_inputs(w, device="cpu", B=8)
    f64 = lambda t: t.to(torch.float64).numpy()
    nbytes, n, t0 = 0, 0, time.perf_counter()
    while n < min(max_seqs, q.shape[0]):
        L = int(lens[n])
        oracle.decode(f64(q[n:n + 1]), f64(kc[n:n + 1, :, :L]), f64(vc[n:n + 1, :, :L]), [L],
                      w.scale)
        nbytes += accounting.decode_kv_bytes([L], w.g, w.d)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return nbytes / dt / 1e9, n, dt


# --------------------------------------------------------------------- native arm

def _step_buffers(w, dev):
    import torch

    from grouped_query_attention_10_b300 import inputs

    q, k, v = inputs.prefill_inputs(w, device=dev)
    return {
        "q": q, "k": k, "v": v,
        "k_new": inputs.random_bf16((w.B, 1, w.g, w.d), 2001, device=dev),
        "v_new": inputs.random_bf16((w.B, 1, w.g, w.d), 2002, device=dev),
        "q_new": inputs.random_bf16((w.B, w.h_q, w.d), 2003, device=dev),
        "lens0": torch.zeros((w.B,), dtype=torch.int32, device=dev),
    }


def native_arm(args):
    import torch

    from grouped_query_attention_10_b300 import accounting, inputs
    from grouped_query_attention_10_b300 import binding as gqa
    from grouped_query_attention_10_b300.run_workload import make_l2_flush

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rank, world = dist_init("nccl")
    gqa.load_library()
    peaks, peak_src = load_peaks()

    w = inputs.LLAMA_CAUSAL_PREFILL
    B, L, h_q, g, d = w.B, w.L, w.h_q, w.g, w.d
    S_max = L + 1
    buf = _step_buffers(w, dev)
    kc = torch.empty((B, g, S_max, d), dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    lens = torch.zeros((B,), dtype=torch.int32, device=dev)
    o = torch.empty((B, L, h_q, d), dtype=torch.bfloat16, device=dev)
    od = torch.empty((B, h_q, d), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(gqa.gqa_decode_workspace_bytes(B, h_q, g, d, S_max), dtype=torch.uint8,
                     device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = make_l2_flush(dev)
    stream = torch.cuda.current_stream(dev)

    flops_prefill = accounting.prefill_flops(B, L, h_q, d, True)
    flops_step = flops_prefill + accounting.decode_flops([S_max] * B, h_q, d)
    # append (rows + lengths), prefill, append (rows + lengths), decode (split + combine)
    launches_per_step = 2 + 1 + 2 + 2

    def step_parts(s, bf, o_out, od_out):
        # the step in three parts, split where the prefill is timed on its own
        def pre():
            lens.zero_()
            gqa.kv_cache_append(kc, vc, lens, bf["k"], bf["v"], status=status, stream=s)

        def pf():
            gqa.gqa_prefill_fwd(bf["q"], bf["k"], bf["v"], causal=True, scale=w.scale,
                                out=o_out, status=status, stream=s)

        def post():
            gqa.kv_cache_append(kc, vc, lens, bf["k_new"], bf["v_new"], status=status, stream=s)
            gqa.gqa_decode_fwd(bf["q_new"], kc, vc, lens, scale=w.scale, out=od_out,
                               workspace=ws, status=status, stream=s)
        return pre, pf, post

    eager_parts = step_parts(stream, buf, o, od)

    def step():
        for fn in eager_parts:
            fn()

    for _ in range(max(args.warmup, 3)):
        flush()
        step()
    torch.cuda.synchronize()
    o_eager, od_eager = o.clone(), od.clone()

    # The timed steps replay the same library calls captured as CUDA graphs
    # (the small append / decode launches then follow each other without host
    # round trips); the results must equal the eager ones bit for bit.
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    graphs = []
    with torch.cuda.stream(cap):
        for fn in step_parts(cap, buf, o, od):
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

    prefill_s = statistics.mean(prefill_ms) / 1e3
    achieved = flops_prefill / prefill_s / 1e12
    roofline = {
        "bound": "tensor", "kernel": "prefill_kernel<128,causal>",
        "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
        "frac": round(achieved / peaks["bf16_tflops"], 4),
        "peak_source": f"{peak_src} bf16 dense burst (cuBLAS)",
        "nominal_peak": NOMINAL_BF16_TFLOPS,
        "frac_of_nominal": round(achieved / NOMINAL_BF16_TFLOPS, 4),
        "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
        "traffic": profiled_traffic("prefill_causal_d128", OUT_DTYPE_NAME),
        "traffic_unit": "bytes per launch (ncu dram read+write)",
        "algorithmic_bytes": accounting.prefill_bytes(B, L, h_q, g, d, o.element_size()),
        "algorithmic_flops": flops_prefill,
        "launch_ms": round(prefill_s * 1e3, 4),
        "timed": f"CUDA events around the prefill inside each of the {args.steps} steps",
    }
    del o_eager, od_eager
    torch.cuda.empty_cache()

    e2e = None
    if not args.step_only:
        roofline["decode"] = decode_roofline(dev, stream, peaks, peak_src, flush)
        torch.cuda.empty_cache()
        e2e = e2e_pipelined(args, dev, w, kc, vc, lens, ws, status, flops_step)
        torch.cuda.empty_cache()

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
        "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": w.name,
                   "B": B, "L": L, "h_q": h_q, "g": g, "d": d, "causal": True,
                   "out": f"{OUT_DTYPE_NAME} (the input dtype; fp32 products, softmax and "
                          "accumulation)",
                   "step": "append prompt K/V, causal prefill, append 1 token, decode 1 token",
                   "flops": "causal pairs only: 4*B*h_q*d*L(L+1)/2 + decode 4*B*h_q*d*(L+1)",
                   "l2": "flushed between timed steps (256 MiB write, then 256 MiB read)",
                   "launch": "each step replays three CUDA graphs of the library calls "
                             "(length reset + prompt append | prefill | token append + decode)",
                   "decode_workload": inputs.DECODE_RAGGED.name,
                   "parallelism": f"replicas x{world}"},
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }

    # the GPU context measurements run before the CPU oracle legs, whose BLAS
    # threads can keep host cores busy (and delay back-to-back launches)
    if not (args.no_extra or args.step_only):
        result["extra"] = extra_measurements(dev, stream, peaks, peak_src, flush)
    if rank == 0 and world == 1 and not args.step_only:
        budget = float(os.environ.get("GQA_BENCH_CPU_BUDGET_S", "12"))
        tf, groups, dt = cpu_oracle_prefill_sample(budget)
        gbs, nseq, dtd = cpu_oracle_decode_sample(budget / 2)
        result["cpu_baseline"] = {
            "value": tf, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "cpu": cpu_model(),
            "sample": f"fp64 NumPy oracle, causal prefill of {groups} of the 32 K/V groups "
                      f"(4 query heads x 4096 rows each, blocks of 512 rows; {dt:.1f} s)",
            "decode": {"value": round(gbs, 4), "unit": "GB/s", "kind": "oracle",
                       "sample": f"fp64 NumPy oracle decode of {nseq} ragged sequences "
                                 f"of the decode workload ({dtd:.1f} s)"},
        }
    if rank == 0:
        print(json.dumps(result), flush=True)


def decode_roofline(dev, stream, peaks, peak_src, flush, n_calls=60):
    """KV-read rate of the ragged decode workload (split + combine launches),
    against the measured HBM copy rate and the nominal HBM figure."""
    import torch

    from grouped_query_attention_10_b300 import accounting, inputs
    from grouped_query_attention_10_b300 import binding as gqa

    w = inputs.DECODE_RAGGED
    q, kc, vc, lens = inputs.decode_inputs(w, device=dev)
    o = torch.empty((w.B, w.h_q, w.d), dtype=torch.float32, device=dev)
    ws = torch.empty(gqa.gqa_decode_workspace_bytes(w.B, w.h_q, w.g, w.d, w.S_max),
                     dtype=torch.uint8, device=dev)
    eager = lambda s_: gqa.gqa_decode_fwd(q, kc, vc, lens, scale=w.scale, out=o, workspace=ws,
                                          stream=s_)
    eager(stream)
    torch.cuda.synchronize()
    o_eager = o.clone()
    # timed as a CUDA graph of the library call (counter reset, split pass,
    # combine), as a serving loop replays it; the replay must match the eager
    # call bit for bit
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            eager(cap)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    if not torch.equal(o, o_eager):
        raise RuntimeError("graph replay of the decode differs from the eager call")
    fn = graph.replay
    _time_calls(fn, 5, stream, flush)
    ts = _time_calls(fn, n_calls, stream, flush)
    ts_eager = _time_calls(lambda: eager(stream), 20, stream, flush)
    nbytes = accounting.decode_kv_bytes(lens.tolist(), w.g, w.d)
    t = statistics.mean(ts)
    gbs = nbytes / t / 1e9
    block = {
        "bound": "hbm", "kernel": "decode_split_kernel<128,1> + decode_combine_kernel<128>",
        "workload": w.name, "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
        "frac": round(gbs / peaks["hbm_gbs"], 4),
        "peak_source": f"{peak_src} HBM copy rate (read+write bytes)",
        "nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4),
        "traffic": profiled_traffic("decode_ragged"),
        "traffic_unit": "bytes per launch of decode_split_kernel (ncu dram read+write)",
        "algorithmic_bytes": nbytes, "launch_us": round(t * 1e6, 2),
        "median_us": round(statistics.median(ts) * 1e6, 2),
        "eager_us": round(statistics.mean(ts_eager) * 1e6, 2),
        "timed": f"CUDA events, mean of {n_calls} replays of a CUDA graph of the call "
                 "(counter reset + split pass + combine), L2 flushed before each",
    }
    return block


def e2e_pipelined(args, dev, w, kc, vc, lens, ws, status, flops_step):
    """The step through the public API with the inputs in pinned host memory
    and the outputs read back every step: host->device copies, the library
    calls and device->host copies run on three streams, two steps in flight."""
    import torch

    from grouped_query_attention_10_b300 import binding as gqa

    B, L, h_q, d = w.B, w.L, w.h_q, w.d
    host_src = _step_buffers(w, "cpu")
    h_in = {k: t.pin_memory() for k, t in host_src.items()}
    d_in = [{k: torch.empty_like(t, device=dev) for k, t in h_in.items()} for _ in range(2)]
    d_o = [torch.empty((B, L, h_q, d), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    d_od = [torch.empty((B, h_q, d), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    h_o = [torch.empty((B, L, h_q, d), dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    h_od = [torch.empty((B, h_q, d), dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = d_o[0].numel() * d_o[0].element_size() + d_od[0].numel() * d_od[0].element_size()
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    in_ready = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    torch.cuda.synchronize()
    for e in comp_done + out_done:
        e.record(s_comp)

    def run(n):
        for i in range(n):
            sl = i % 2
            s_in.wait_event(comp_done[sl])  # step i-2 no longer reads this slot's inputs
            with torch.cuda.stream(s_in):
                for k, t in h_in.items():
                    d_in[sl][k].copy_(t, non_blocking=True)
            in_ready[sl].record(s_in)
            s_comp.wait_event(in_ready[sl])
            s_comp.wait_event(out_done[sl])  # step i-2's outputs have been read back
            bf = d_in[sl]
            with torch.cuda.stream(s_comp):
                lens.copy_(bf["lens0"], non_blocking=True)
            gqa.kv_cache_append(kc, vc, lens, bf["k"], bf["v"], status=status, stream=s_comp)
            gqa.gqa_prefill_fwd(bf["q"], bf["k"], bf["v"], causal=True, scale=w.scale,
                                out=d_o[sl], status=status, stream=s_comp)
            gqa.kv_cache_append(kc, vc, lens, bf["k_new"], bf["v_new"], status=status,
                                stream=s_comp)
            gqa.gqa_decode_fwd(bf["q_new"], kc, vc, lens, scale=w.scale, out=d_od[sl],
                               workspace=ws, status=status, stream=s_comp)
            comp_done[sl].record(s_comp)
            s_out.wait_event(comp_done[sl])
            with torch.cuda.stream(s_out):
                h_o[sl].copy_(d_o[sl], non_blocking=True)
                h_od[sl].copy_(d_od[sl], non_blocking=True)
            out_done[sl].record(s_out)

    run(3)
    torch.cuda.synchronize()
    n = max(args.steps // 4, 8)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    t0.record(s_in)
    run(n)
    s_out.wait_stream(s_in)
    s_out.wait_stream(s_comp)
    t1.record(s_out)
    torch.cuda.synchronize()
    e2e_t = reduce_max(t0.elapsed_time(t1) / 1e3, dev)
    units = reduce_sum(flops_step * n, dev)
    return {"value": round(units / e2e_t / 1e12, 3), "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(e2e_t * 1e3 / n, 4), "steps": n,
            "how": "public API calls on a compute stream; pinned host->device copies of each "
                   "step's inputs and device->host copies of O and the decode output on two "
                   "copy streams, two steps in flight"}


def extra_measurements(dev, stream, peaks, peak_src, flush):
    """Context measurements on the other workloads (not part of `value`)."""
    import torch

    from grouped_query_attention_10_b300 import run_workload

    out = {}

    def one(name, n=20, peak=None, nominal=None):
        fn, work, unit, div = run_workload.make(name, dev)
        call = lambda: fn(stream)
        reset = getattr(fn, "reset", None)  # an append's empty-cache reset, untimed
        prep = flush if reset is None else (lambda: (reset(), flush()))
        _time_calls(call, 3, stream, prep)
        ts = _time_calls(call, n, stream, prep)
        # the median call (a context figure robust to an occasional slow call);
        # the mean beside it
        t = statistics.median(ts)
        rate = work / t / div
        rec = {"rate": round(rate, 2), "unit": unit, "us": round(t * 1e6, 2),
               "mean_us": round(statistics.mean(ts) * 1e6, 2), "timed": f"median of {n} calls"}
        if unit == "TFLOP/s":
            rec["frac_of_bf16_peak"] = round(rate / peaks["bf16_tflops"], 4)
            rec["frac_of_nominal"] = round(rate / NOMINAL_BF16_TFLOPS, 4)
        else:
            rec["frac_of_hbm"] = round(rate / peaks["hbm_gbs"], 4)
            rec["frac_of_nominal"] = round(rate / NOMINAL_HBM_GBS, 4)
        rec["peak_source"] = peak_src
        del fn
        torch.cuda.empty_cache()
        return rec

    out["prefill_noncausal_b32_l1024_hq8_g4_d64"] = one("prefill_noncausal", 50)
    # the headline prefill with fp32 output instead of the step's bf16
    out["prefill_causal_fp32_output"] = one("prefill_causal", 20)
    for g in (1, 2, 4, 8, 16, 32):
        out[f"decode_sweep_b16_hq32_g{g}_d128_s32768"] = one(f"decode_sweep_g{g}", 20)
    for name in ("prefill_window", "prefill_alibi", "prefill_kvcache", "decode_paged_p16",
                 "decode_paged_p64", "decode_window", "append_prompt", "append_rope"):
        out[name] = one(name, 20)
    # the prefill workloads above write fp32 output; the same with bf16 output
    # (the input dtype, as in the step)
    for name in ("prefill_noncausal_bf16", "prefill_window_bf16", "prefill_alibi_bf16",
                 "prefill_kvcache_bf16"):
        out[name] = one(name, 20)
    return out


# --------------------------------------------------------------------- reference arm

def reference_arm(args):
    """The CPU oracle, timed as it stands, on bounded samples of the workload:
    each step is one block of 256 query rows of one causal K/V group."""
    from grouped_query_attention_10_b300 import inputs

    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = inputs.LLAMA_CAUSAL_PREFILL
    G = w.h_q // w.g
    rows = 256
    q, k, v = inputs.prefill_inputs(w, device="cpu", B=1)
    groups = [_group_slice(q, k, v, 0, kvh, G) for kvh in range(2)]
    blocks = [(gi, r0) for gi in range(len(groups)) for r0 in range(0, w.L, rows)]

    def step(i):
        gi, r0 = blocks[i % len(blocks)]
        qs, ks, vs = groups[gi]
        return oracle_prefill_block(qs, ks, vs, r0, rows, w.scale)

    for i in range(max(args.warmup, 1)):
        step(i)
    t0 = time.perf_counter()
    flops = 0
    for i in range(args.steps):
        flops += step(i)
    dt = time.perf_counter() - t0
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
        "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": w.name, "B": w.B, "L": w.L, "h_q": w.h_q, "g": w.g, "d": w.d,
                   "causal": True, "out": "f64 (the oracle)", "parallelism": "cpu, rank 0 only"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(),
                         "kind": "oracle", "cpu": cpu_model(),
                         "sample": f"fp64 NumPy oracle, one block of {rows} causal query rows "
                                   f"of one K/V group ({G} query heads) per step, cycling "
                                   "over the rows of two groups"},
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
