"""Run one named GQA workload on the GPU and report its kernel time.

    python -m grouped_query_attention_10_b300.run_workload <name> [--iters N] [--warmup W]

Names: prefill_tiny, prefill_noncausal, prefill_causal (fp32 output),
prefill_causal_bf16 (bf16 output, as in the bench step), decode_ragged,
decode_sweep_g{1,2,4,8,16,32}, append_prompt, and the variants prefill_window
(W = 1024), prefill_alibi, prefill_kvcache (512 new tokens over 4096),
decode_paged_p{16,64,256}, decode_window (W = 1024), append_rope. Inputs are the seeded
synthetic workloads of ``inputs.py``. The prefill workloads write fp32 output;
prefill_{noncausal,window,alibi,kvcache}_bf16 are the same with bf16 output.
Each timed call is bracketed by CUDA
events on the launching stream; an L2 flush precedes every call (a 256 MiB
write, then a 256 MiB read of another buffer, so the write's dirty lines are
written back before the timed call starts). The append workloads write into
an empty cache every call: their length reset (``fn.reset``) runs before the
flush, outside the timed interval. Handy for profiling one kernel in
isolation.
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


def _prefill(w, dev, B=None, out_dtype=torch.float32):
    if B is not None:
        w = dataclasses.replace(w, B=B)
    q, k, v = inputs.prefill_inputs(w, device=dev)
    o = torch.empty((w.B, w.L, w.h_q, w.d), dtype=out_dtype, device=dev)
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
        gqa.kv_cache_append(kc, vc, lens, k, v, stream=s)

    fn.reset = lens.zero_
    return fn, accounting.append_bytes(w.B, w.L, w.g, w.d), "GB/s", 1e9


def _prefill_variant(dev, window=0, alibi=False, out_dtype=torch.float32):
    """The causal Llama-shape prefill with a sliding window or ALiBi slopes."""
    w = inputs.LLAMA_CAUSAL_PREFILL
    q, k, v = inputs.prefill_inputs(w, device=dev)
    o = torch.empty((w.B, w.L, w.h_q, w.d), dtype=out_dtype, device=dev)
    slopes = (torch.tensor([2.0 ** (-8.0 * (h + 1) / w.h_q) for h in range(w.h_q)],
                           dtype=torch.float32, device=dev) if alibi else None)
    fn = lambda s: gqa.gqa_prefill_fwd(q, k, v, causal=True, scale=w.scale, out=o, stream=s,
                                       window=window, alibi_slopes=slopes)
    work = (accounting.prefill_window_flops(w.B, w.L, w.h_q, w.d, window) if window
            else accounting.prefill_flops(w.B, w.L, w.h_q, w.d, True))
    return fn, work, "TFLOP/s", 1e12


def _prefill_kvcache(dev, T=512, out_dtype=torch.float32):
    """Chunked prefill: the last T of 4096 tokens per sequence of the Llama
    shape attend to the whole cache."""
    w = inputs.LLAMA_CAUSAL_PREFILL
    q, k, v = inputs.prefill_inputs(w, device=dev)
    kc = k.transpose(1, 2).contiguous()
    vc = v.transpose(1, 2).contiguous()
    qn = q[:, w.L - T:].contiguous()
    lens = torch.full((w.B,), w.L, dtype=torch.int32, device=dev)
    o = torch.empty((w.B, T, w.h_q, w.d), dtype=out_dtype, device=dev)
    fn = lambda s: gqa.gqa_prefill_kvcache_fwd(qn, kc, vc, lens, scale=w.scale, out=o, stream=s)
    return fn, accounting.prefill_cached_flops([w.L] * w.B, T, w.h_q, w.d), "TFLOP/s", 1e12


def _decode_paged(dev, page):
    """The ragged decode workload through a paged pool (shuffled pages)."""
    w = inputs.DECODE_RAGGED
    q, kc, vc, lens = inputs.decode_inputs(w, device=dev)
    nb = w.S_max // page
    perm = torch.randperm(w.B * nb, generator=torch.Generator().manual_seed(page))
    pool_of = lambda c: c.view(w.B, w.g, nb, page, w.d).permute(0, 2, 1, 3, 4).reshape(
        w.B * nb, w.g, page, w.d)
    kp = torch.empty_like(kc).view(w.B * nb, w.g, page, w.d)
    vp = torch.empty_like(kp)
    kp[perm.to(dev)] = pool_of(kc)
    vp[perm.to(dev)] = pool_of(vc)
    table = perm.view(w.B, nb).to(torch.int32).to(dev)
    del kc, vc
    o = torch.empty((w.B, w.h_q, w.d), dtype=torch.float32, device=dev)
    ws = torch.empty(gqa.gqa_decode_paged_workspace_bytes(w.B, w.h_q, w.g, w.d, page, nb),
                     dtype=torch.uint8, device=dev)
    fn = lambda s: gqa.gqa_decode_paged_fwd(q, kp, vp, table, lens, scale=w.scale, out=o,
                                            workspace=ws, stream=s)
    return fn, accounting.decode_kv_bytes(lens.tolist(), w.g, w.d), "GB/s", 1e9


def _decode_window(dev, window=1024):
    """The ragged decode workload with a sliding window."""
    w = inputs.DECODE_RAGGED
    q, kc, vc, lens = inputs.decode_inputs(w, device=dev)
    o = torch.empty((w.B, w.h_q, w.d), dtype=torch.float32, device=dev)
    ws = torch.empty(gqa.gqa_decode_workspace_bytes(w.B, w.h_q, w.g, w.d, w.S_max),
                     dtype=torch.uint8, device=dev)
    fn = lambda s: gqa.gqa_decode_fwd(q, kc, vc, lens, scale=w.scale, out=o, workspace=ws,
                                      stream=s, window=window)
    return fn, accounting.decode_window_kv_bytes(lens.tolist(), window, w.g, w.d), "GB/s", 1e9


def _append_rope(dev):
    """The bench step's prompt (B32 T1024 h8 g4 d64) through the fused RoPE append."""
    w = inputs.NONCAUSAL_PREFILL
    q, k, v = inputs.prefill_inputs(w, device=dev)
    kc = torch.empty((w.B, w.g, w.L, w.d), dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    qo = torch.empty_like(q)
    lens = torch.zeros((w.B,), dtype=torch.int32, device=dev)
    ang = torch.arange(w.L, dtype=torch.float64)[:, None] * 10000.0 ** (
        -torch.arange(0, w.d, 2, dtype=torch.float64) / w.d)[None, :]
    cos = torch.cos(ang).float().to(dev)
    sin = torch.sin(ang).float().to(dev)

    def fn(s):
        gqa.kv_cache_append_rope(kc, vc, lens, k, v, cos, sin, q=q, q_out=qo, stream=s)

    fn.reset = lens.zero_
    return fn, accounting.rope_append_bytes(w.B, w.L, w.h_q, w.g, w.d), "GB/s", 1e9


def make(name: str, dev, B=None):
    if name.endswith("_bf16") and name != "prefill_causal_bf16":
        # the same workload with bf16 output (the input dtype)
        base = name[:-len("_bf16")]
        bf = torch.bfloat16
        if base == "prefill_noncausal":
            return _prefill(inputs.NONCAUSAL_PREFILL, dev, B, out_dtype=bf)
        if base == "prefill_window":
            return _prefill_variant(dev, window=1024, out_dtype=bf)
        if base == "prefill_alibi":
            return _prefill_variant(dev, alibi=True, out_dtype=bf)
        if base == "prefill_kvcache":
            return _prefill_kvcache(dev, out_dtype=bf)
        raise SystemExit(f"unknown workload {name}")
    if name == "prefill_tiny":
        return _prefill(inputs.TINY_CAUSAL_PREFILL, dev, B)
    if name == "prefill_noncausal":
        return _prefill(inputs.NONCAUSAL_PREFILL, dev, B)
    if name == "prefill_causal":
        return _prefill(inputs.LLAMA_CAUSAL_PREFILL, dev, B)
    if name == "prefill_causal_bf16":
        return _prefill(inputs.LLAMA_CAUSAL_PREFILL, dev, B, out_dtype=torch.bfloat16)
    if name == "decode_ragged":
        return _decode(inputs.DECODE_RAGGED, dev, B)
    if name.startswith("decode_sweep_g"):
        return _decode(inputs.decode_sweep(int(name[len("decode_sweep_g"):])), dev, B)
    if name == "append_prompt":
        return _append(dev)
    if name == "prefill_window":
        return _prefill_variant(dev, window=1024)
    if name == "prefill_alibi":
        return _prefill_variant(dev, alibi=True)
    if name == "prefill_kvcache":
        return _prefill_kvcache(dev)
    if name.startswith("decode_paged_p"):
        return _decode_paged(dev, int(name[len("decode_paged_p"):]))
    if name == "decode_window":
        return _decode_window(dev)
    if name == "append_rope":
        return _append_rope(dev)
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
    reset = getattr(fn, "reset", lambda: None)
    for _ in range(a.warmup):
        reset()
        flush()
        fn(s)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(a.iters)]
    for e0, e1 in evs:
        reset()
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
