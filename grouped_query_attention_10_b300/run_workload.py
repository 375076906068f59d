"""Run one named GQA workload on the GPU and report its kernel time.

    python -m grouped_query_attention_10_b300.run_workload <name> [--iters N] [--warmup W]

Names: prefill_tiny, prefill_noncausal, prefill_causal, decode_ragged,
decode_sweep_g{1,2,4,8,16,32}, append_prompt. Inputs are the seeded
synthetic workloads of ``inputs.py``. Each timed call is bracketed by CUDA
events on the launching stream; an L2 flush precedes every call (a 256 MiB
write, then a 256 MiB read of another buffer, so the write's dirty lines are
written back before the timed call starts). Handy for profiling one kernel
in isolation.
"""

from __future__ import annotations

import argparse
import dataclasses
import json
import statistics

import torch

from . import accounting, inputs
from . import binding as gqa

L2_FLUSH_BYTES = 256 << 20


def make_l2_flush(dev):
    """Return a function that leaves no input and no dirty line in L2 (126 MB
    on B300): write a buffer larger than L2, then read another one."""
    wbuf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    rbuf = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush():
        wbuf.fill_(1)
        rbuf.sum()

    return flush


def _prefill(w, dev, B=None):
    if B is not None:
        w = dataclasses.replace(w, B=B)
    q, k, v = inputs.prefill_inputs(w, device=dev)
    o = torch.empty((w.B, w.L, w.h_q, w.d), dtype=torch.float32, device=dev)
    fn = lambda s: gqa.gqa_prefill_fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, stream=s)
    work = accounting.prefill_flops(w.B, w.L, w.h_q, w.d, w.causal)
    return fn, work, "TFLOP/s", 1e12


def _decode(w, dev, B=None):
    if B is not None:
        w = dataclasses.replace(w, B=B)
    q, kc, vc, lens = inputs.decode_inputs(w, device=dev)
    o = torch.empty((w.B, w.h_q, w.d), dtype=torch.float32, device=dev)
    ws = torch.empty(gqa.gqa_decode_workspace_bytes(w.B, w.h_q, w.g, w.d, w.S_max),
                     dtype=torch.uint8, device=dev)
    fn = lambda s: gqa.gqa_decode_fwd(q, kc, vc, lens, scale=w.scale, out=o, workspace=ws,
                                      stream=s)
    work = accounting.decode_kv_bytes(lens.tolist(), w.g, w.d)
    return fn, work, "GB/s", 1e9


def _append(dev):
    w = inputs.NONCAUSAL_PREFILL
    _, k, v = inputs.prefill_inputs(w, device=dev)
    kc = torch.empty((w.B, w.g, w.L, w.d), dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    lens = torch.zeros((w.B,), dtype=torch.int32, device=dev)

    def fn(s):
        lens.zero_()
        gqa.kv_cache_append(kc, vc, lens, k, v, stream=s)

    return fn, accounting.append_bytes(w.B, w.L, w.g, w.d), "GB/s", 1e9


def make(name: str, dev, B=None):
    if name == "prefill_tiny":
        return _prefill(inputs.TINY_CAUSAL_PREFILL, dev, B)
    if name == "prefill_noncausal":
        return _prefill(inputs.NONCAUSAL_PREFILL, dev, B)
    if name == "prefill_causal":
        return _prefill(inputs.LLAMA_CAUSAL_PREFILL, dev, B)
    if name == "decode_ragged":
        return _decode(inputs.DECODE_RAGGED, dev, B)
    if name.startswith("decode_sweep_g"):
        return _decode(inputs.decode_sweep(int(name[len("decode_sweep_g"):])), dev, B)
    if name == "append_prompt":
        return _append(dev)
    raise SystemExit(f"unknown workload {name}")


def main(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("name")
    p.add_argument("--iters", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--batch", type=int, default=None, help="override the workload's B")
    a = p.parse_args(argv)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    fn, work, unit, div = make(a.name, dev, a.batch)
    s = torch.cuda.current_stream(dev)
    flush = make_l2_flush(dev)
    for _ in range(a.warmup):
        flush()
        fn(s)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(a.iters)]
    for e0, e1 in evs:
        flush()
        e0.record(s)
        fn(s)
        e1.record(s)
    torch.cuda.synchronize()
    ts = [e0.elapsed_time(e1) / 1e3 for e0, e1 in evs]
    t = statistics.median(ts)
    print(json.dumps({"workload": a.name, "batch": a.batch, "median_us": round(t * 1e6, 2),
                      "rate": round(work / t / div, 2), "unit": unit, "iters": a.iters}))


if __name__ == "__main__":
    main()
