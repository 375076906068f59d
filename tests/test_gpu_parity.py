"""GPU parity: the CUDA path (through the C interface) against the fp64 oracle.

Inputs are seeded bf16 tensors; the oracle reads the very same bf16 values
(copied back from the device). Tolerance for floating-point outputs: max
abs error <= 1e-2 and mean abs error <= 1e-3 (fp32 accumulation, bf16
probabilities); the KV-cache append must be bit exact.

Small sizes are compared element by element; the full-size workloads run in
the same launch configuration the benchmark times and are checked on sampled
output rows that the oracle computes one by one.

Output, lse and cache buffers sit between NaN guard bands (tests/guard.py);
every call must leave the bands untouched and must write every element of its
outputs (they start as NaN).
"""

import math

import numpy as np
import pytest
import torch

import guard
import oracle
from grouped_query_attention_10_b300 import binding as gqa
from grouped_query_attention_10_b300 import inputs

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-2
MEAN_ABS = 1e-3
DEV = "cuda"


def f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def assert_close(got, ref, what, max_abs=MAX_ABS, mean_abs=MEAN_ABS):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    assert err.max() <= max_abs, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= mean_abs, f"{what}: mean abs err {err.mean():.3e}"


def rand_bf16(shape, seed):
    return inputs.random_bf16(shape, seed, device="cpu").to(DEV)


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------

def run_prefill(B, L, h_q, g, d, causal, seed, out_dtype=torch.float32, with_lse=True):
    q = rand_bf16((B, L, h_q, d), seed)
    k = rand_bf16((B, L, g, d), seed + 1)
    v = rand_bf16((B, L, g, d), seed + 2)
    scale = 1.0 / math.sqrt(d)
    go = guard.empty((B, L, h_q, d), out_dtype, DEV)
    gl = guard.empty((B, h_q, L), torch.float32, DEV) if with_lse else None
    lse = gl.tensor if with_lse else None
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = gqa.gqa_prefill_fwd(q, k, v, causal=causal, scale=scale, out=go.tensor, lse=lse,
                            status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    go.assert_bands(f"prefill O B={B} L={L} d={d}")
    if with_lse:
        gl.assert_bands(f"prefill lse B={B} L={L} d={d}")
    o_ref, lse_ref = oracle.prefill(f64(q), f64(k), f64(v), causal, scale)
    return o, lse, o_ref, lse_ref


def test_prefill_tiny_causal_workload():
    w = inputs.TINY_CAUSAL_PREFILL
    q, k, v = (t.to(DEV) for t in inputs.prefill_inputs(w))
    lse = torch.empty((w.B, w.h_q, w.L), dtype=torch.float32, device=DEV)
    o = gqa.gqa_prefill_fwd(q, k, v, causal=True, scale=w.scale, lse=lse)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.prefill(f64(q), f64(k), f64(v), True, w.scale)
    assert_close(f64(o), o_ref, "tiny causal prefill O")
    assert_close(f64(lse), lse_ref, "tiny causal prefill lse")
    # causal row 0 returns V[0] of its K/V head (up to bf16 rounding of P = 1)
    kvh = np.arange(w.h_q) // (w.h_q // w.g)
    np.testing.assert_allclose(f64(o)[:, 0], f64(v)[:, 0, kvh, :], rtol=0, atol=1e-6)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("L", [1, 63, 127, 129, 200, 384])
def test_prefill_ragged_lengths(d, causal, L):
    o, lse, o_ref, lse_ref = run_prefill(2, L, 8, 2, d, causal, seed=100 + L + d)
    assert_close(f64(o), o_ref, f"prefill L={L} d={d} causal={causal}")
    assert_close(f64(lse), lse_ref, "lse")


@pytest.mark.parametrize("h_q,g", [(4, 4), (8, 4), (8, 2), (16, 2), (32, 2), (32, 1),
                                   (64, 1), (128, 1)])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("d", [64, 128])
def test_prefill_group_sizes(h_q, g, causal, d):
    o, lse, o_ref, lse_ref = run_prefill(1, 160, h_q, g, d, causal, seed=7 * h_q + g + d)
    assert_close(f64(o), o_ref, f"prefill h_q={h_q} g={g}")
    assert_close(f64(lse), lse_ref, "lse")


@pytest.mark.parametrize("d,causal", [(128, True), (64, False), (128, False)])
def test_prefill_bf16_output(d, causal):
    o, _, o_ref, _ = run_prefill(1, 256, 8, 2, d, causal, seed=31 + d, out_dtype=torch.bfloat16,
                                 with_lse=False)
    assert o.dtype == torch.bfloat16
    # the same bounds as the fp32 output, against the unrounded fp64 oracle
    assert_close(f64(o), o_ref, f"prefill bf16 out d={d} causal={causal}")


def test_prefill_noncausal_workload_reduced_batch():
    w = inputs.NONCAUSAL_PREFILL
    q, k, v = (t.to(DEV) for t in inputs.prefill_inputs(w, B=2))
    o = gqa.gqa_prefill_fwd(q, k, v, causal=False, scale=w.scale)
    torch.cuda.synchronize()
    o_ref, _ = oracle.prefill(f64(q), f64(k), f64(v), False, w.scale)
    assert_close(f64(o), o_ref, "non-causal prefill, 2 sequences")


def test_prefill_llama_causal_reduced_length():
    w = inputs.LLAMA_CAUSAL_PREFILL
    q, k, v = (t.to(DEV) for t in inputs.prefill_inputs(w, B=1, L=1024))
    o = gqa.gqa_prefill_fwd(q, k, v, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    o_ref, _ = oracle.prefill(f64(q), f64(k), f64(v), True, w.scale)
    assert_close(f64(o), o_ref, "llama causal prefill, L=1024")


def _sampled_prefill_check(w, n_rows, seed, out_dtype=torch.float32):
    q, k, v = inputs.prefill_inputs(w, device=DEV)
    lse = torch.empty((w.B, w.h_q, w.L), dtype=torch.float32, device=DEV)
    o = gqa.gqa_prefill_fwd(q, k, v, causal=w.causal, scale=w.scale, lse=lse, out_dtype=out_dtype)
    torch.cuda.synchronize()
    rng = np.random.default_rng(seed)
    rows = [(int(rng.integers(w.B)), int(rng.integers(w.L))) for _ in range(n_rows)]
    rows += [(0, 0), (w.B - 1, w.L - 1)]
    got, ref, got_l, ref_l = [], [], [], []
    for b, pos in rows:
        kv_len = pos + 1 if w.causal else w.L
        o_r, l_r = oracle.prefill(f64(q[b:b + 1, pos:pos + 1]), f64(k[b:b + 1, :kv_len]),
                                  f64(v[b:b + 1, :kv_len]), w.causal, w.scale, q_offset=pos)
        got.append(f64(o[b, pos]))
        ref.append(o_r[0, 0])
        got_l.append(f64(lse[b, :, pos]))
        ref_l.append(l_r[0, :, 0])
    assert_close(np.stack(got), np.stack(ref), f"{w.name} sampled rows")
    assert_close(np.stack(got_l), np.stack(ref_l), f"{w.name} sampled lse")


def test_prefill_noncausal_workload_full_size_sampled():
    _sampled_prefill_check(inputs.NONCAUSAL_PREFILL, 24, seed=5)


def test_prefill_llama_causal_workload_full_size_sampled():
    _sampled_prefill_check(inputs.LLAMA_CAUSAL_PREFILL, 24, seed=6)


def test_prefill_llama_causal_workload_full_size_sampled_bf16_output():
    # the launch configuration the bench step times: bf16 output (the input
    # dtype), fp32 accumulation; the output's own rounding is inside the bound
    _sampled_prefill_check(inputs.LLAMA_CAUSAL_PREFILL, 24, seed=7, out_dtype=torch.bfloat16)


# ---------------------------------------------------------------------------
# decode
# ---------------------------------------------------------------------------

def run_decode(q, kc, vc, lens, scale, out_dtype=torch.float32):
    gl = guard.empty(tuple(q.shape[:2]), torch.float32, DEV)
    go = guard.empty(tuple(q.shape), out_dtype, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = gqa.gqa_decode_fwd(q, kc, vc, lens, scale=scale, lse=gl.tensor, out=go.tensor,
                           status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    go.assert_bands("decode O")
    gl.assert_bands("decode lse")
    return o, gl.tensor


def test_decode_ragged_lengths_reduced():
    w = inputs.DECODE_RAGGED
    q, kc, vc, lens = (t.to(DEV) for t in inputs.decode_inputs(w, B=8, S_max=2048))
    lens[:4] = torch.tensor([1, 2, 127, 2048], dtype=torch.int32)
    o, lse = run_decode(q, kc, vc, lens, w.scale)
    o_ref, lse_ref = oracle.decode(f64(q), f64(kc), f64(vc), lens.cpu().numpy(), w.scale)
    assert_close(f64(o), o_ref, "decode ragged")
    assert_close(f64(lse), lse_ref, "decode lse")


@pytest.mark.parametrize("g", inputs.DECODE_SWEEP_G)
def test_decode_group_sweep_reduced(g):
    w = inputs.decode_sweep(g)
    q, kc, vc, lens = (t.to(DEV) for t in inputs.decode_inputs(w, B=2, S_max=3000))
    lens[1] = 1777
    o, lse = run_decode(q, kc, vc, lens, w.scale)
    o_ref, lse_ref = oracle.decode(f64(q), f64(kc), f64(vc), lens.cpu().numpy(), w.scale)
    assert_close(f64(o), o_ref, f"decode g={g}")
    assert_close(f64(lse), lse_ref, f"decode lse g={g}")


def test_decode_ignores_garbage_past_length_and_empty_sequences():
    B, h_q, g, d, S = 3, 16, 4, 128, 700
    q = rand_bf16((B, h_q, d), 41)
    kc = rand_bf16((B, g, S, d), 42)
    vc = rand_bf16((B, g, S, d), 43)
    lens = torch.tensor([333, 0, 700], dtype=torch.int32, device=DEV)
    o_clean, lse_clean = run_decode(q, kc, vc, lens, 0.09)
    kc[0, :, 333:] = float("nan")
    vc[0, :, 333:] = float("inf")
    kc[1] = float("nan")
    vc[1] = float("nan")
    o, lse = run_decode(q, kc, vc, lens, 0.09)
    assert torch.equal(o[0], o_clean[0]) and torch.equal(o[2], o_clean[2])
    assert torch.all(o[1] == 0) and torch.all(torch.isneginf(lse[1]))
    o_ref, lse_ref = oracle.decode(f64(q), f64(kc), f64(vc), lens.cpu().numpy(), 0.09)
    assert_close(f64(o), o_ref, "decode with garbage rows")


def test_decode_bf16_output():
    q = rand_bf16((2, 32, 128), 51)
    kc = rand_bf16((2, 8, 1000, 128), 52)
    vc = rand_bf16((2, 8, 1000, 128), 53)
    lens = torch.tensor([1000, 517], dtype=torch.int32, device=DEV)
    o, _ = run_decode(q, kc, vc, lens, 0.0884, out_dtype=torch.bfloat16)
    o_ref, _ = oracle.decode(f64(q), f64(kc), f64(vc), lens.cpu().numpy(), 0.0884)
    assert o.dtype == torch.bfloat16
    assert_close(f64(o), o_ref, "decode bf16 out")


def test_decode_d64_and_large_group():
    q = rand_bf16((2, 64, 64), 61)
    kc = rand_bf16((2, 1, 900, 64), 62)
    vc = rand_bf16((2, 1, 900, 64), 63)
    lens = torch.tensor([900, 65], dtype=torch.int32, device=DEV)
    o, lse = run_decode(q, kc, vc, lens, 0.125)   # G = 64: two 32-row slices
    o_ref, lse_ref = oracle.decode(f64(q), f64(kc), f64(vc), lens.cpu().numpy(), 0.125)
    assert_close(f64(o), o_ref, "decode d=64 G=64")
    assert_close(f64(lse), lse_ref, "decode lse d=64 G=64")


def test_decode_equals_row_of_causal_prefill_on_gpu():
    B, L, h_q, g, d = 2, 300, 32, 8, 128
    q = rand_bf16((B, L, h_q, d), 71)
    k = rand_bf16((B, L, g, d), 72)
    v = rand_bf16((B, L, g, d), 73)
    lse_p = torch.empty((B, h_q, L), dtype=torch.float32, device=DEV)
    o_p = gqa.gqa_prefill_fwd(q, k, v, causal=True, scale=0.0884, lse=lse_p)
    kc = k.transpose(1, 2).contiguous()
    vc = v.transpose(1, 2).contiguous()
    for t in (0, 1, 150, L - 1):
        lens = torch.full((B,), t + 1, dtype=torch.int32, device=DEV)
        o_d, lse_d = run_decode(q[:, t].contiguous(), kc, vc, lens, 0.0884)
        assert_close(f64(o_d), f64(o_p[:, t]), f"decode vs prefill row {t}", max_abs=5e-3)
        assert_close(f64(lse_d), f64(lse_p[:, :, t]), f"lse row {t}", max_abs=5e-3)


def _sampled_decode_check(w, n_seq, seed):
    q, kc, vc, lens = inputs.decode_inputs(w, device=DEV)
    o, lse = run_decode(q, kc, vc, lens, w.scale)
    rng = np.random.default_rng(seed)
    bs = sorted(set([0, w.B - 1] + [int(x) for x in rng.integers(0, w.B, n_seq)]))
    for b in bs:
        n = int(lens[b].item())
        o_r, l_r = oracle.decode(f64(q[b:b + 1]), f64(kc[b:b + 1, :, :n]),
                                 f64(vc[b:b + 1, :, :n]), [n], w.scale)
        assert_close(f64(o[b:b + 1]), o_r, f"{w.name} sequence {b}")
        assert_close(f64(lse[b:b + 1]), l_r, f"{w.name} lse {b}")


def test_decode_ragged_workload_full_size_sampled():
    _sampled_decode_check(inputs.DECODE_RAGGED, 4, seed=8)


@pytest.mark.parametrize("g", inputs.DECODE_SWEEP_G)
def test_decode_sweep_workload_full_size_sampled(g):
    _sampled_decode_check(inputs.decode_sweep(g), 1, seed=9)
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# KV-cache append
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T", [1, 5, 64])
def test_append_bit_exact(T):
    B, g, S, d = 4, 8, 300, 128
    kc = rand_bf16((B, g, S, d), 81)
    vc = rand_bf16((B, g, S, d), 82)
    kn = rand_bf16((B, T, g, d), 83)
    vn = rand_bf16((B, T, g, d), 84)
    lens = torch.tensor([0, 17, 200, S - T], dtype=torch.int32, device=DEV)
    bits = lambda t: t.view(torch.int16).cpu().numpy()
    k_ref, v_ref, lens_ref, st_ref = oracle.append(bits(kc), bits(vc), lens.cpu().numpy(),
                                                   bits(kn), bits(vn))
    gk, gv, glen = guard.copy_of(kc), guard.copy_of(vc), guard.copy_of(lens)
    kc, vc, lens = gk.tensor, gv.tensor, glen.tensor
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gqa.kv_cache_append(kc, vc, lens, kn, vn, status=status)
    torch.cuda.synchronize()
    for gb, what in ((gk, "K cache"), (gv, "V cache"), (glen, "lengths")):
        gb.assert_bands(f"append T={T} {what}")
    assert np.array_equal(bits(kc), k_ref)
    assert np.array_equal(bits(vc), v_ref)
    assert np.array_equal(lens.cpu().numpy(), lens_ref)
    assert int(status.item()) == st_ref == 0


def test_append_overflow_is_dropped_and_flagged():
    B, g, S, d, T = 2, 2, 40, 64, 8
    kc = torch.zeros((B, g, S, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    kn = rand_bf16((B, T, g, d), 91)
    vn = rand_bf16((B, T, g, d), 92)
    lens = torch.tensor([35, 3], dtype=torch.int32, device=DEV)
    bits = lambda t: t.view(torch.int16).cpu().numpy()
    k_ref, v_ref, lens_ref, st_ref = oracle.append(bits(kc), bits(vc), lens.cpu().numpy(),
                                                   bits(kn), bits(vn))
    gk, gv = guard.copy_of(kc), guard.copy_of(vc)
    kc, vc = gk.tensor, gv.tensor
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gqa.kv_cache_append(kc, vc, lens, kn, vn, status=status)
    torch.cuda.synchronize()
    gk.assert_bands("overflowing append K cache")
    gv.assert_bands("overflowing append V cache")
    assert np.array_equal(bits(kc), k_ref) and np.array_equal(bits(vc), v_ref)
    assert list(lens.cpu().numpy()) == list(lens_ref) == [40, 11]
    assert int(status.item()) == st_ref == oracle.APPEND_CACHE_FULL


def test_append_then_decode_matches_oracle():
    B, h_q, g, d, S = 3, 32, 8, 128, 2048
    kc = rand_bf16((B, g, S, d), 101)
    vc = rand_bf16((B, g, S, d), 102)
    lens = torch.tensor([1000, 2047, 5], dtype=torch.int32, device=DEV)
    kn = rand_bf16((B, 1, g, d), 103)
    vn = rand_bf16((B, 1, g, d), 104)
    q = rand_bf16((B, h_q, d), 105)
    bits = lambda t: t.view(torch.int16).cpu().numpy()
    k_ref, v_ref, lens_ref, _ = oracle.append(bits(kc), bits(vc), lens.cpu().numpy(),
                                              bits(kn), bits(vn))
    gqa.kv_cache_append(kc, vc, lens, kn, vn)
    o, _ = run_decode(q, kc, vc, lens, 0.0884)
    o_ref, _ = oracle.decode(f64(q), oracle.bf16_bits_to_f64(k_ref.view(np.uint16)),
                             oracle.bf16_bits_to_f64(v_ref.view(np.uint16)), lens_ref, 0.0884)
    assert_close(f64(o), o_ref, "append then decode")


def test_append_full_size_decode_workload():
    """One decode-step append on the [64, 8, 8192, 128] cache, bit exact on
    the rows it touches and untouched everywhere else."""
    w = inputs.DECODE_RAGGED
    q, kc, vc, lens = inputs.decode_inputs(w, device=DEV)
    lens[0] = w.S_max  # full: its row must be dropped
    kn = inputs.random_bf16((w.B, 1, w.g, w.d), 111, device=DEV)
    vn = inputs.random_bf16((w.B, 1, w.g, w.d), 112, device=DEV)
    k_before = kc.clone()
    lens_before = lens.clone()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gqa.kv_cache_append(kc, vc, lens, kn, vn, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == oracle.APPEND_CACHE_FULL
    lb = lens_before.long()
    expect = torch.minimum(lb + 1, torch.full_like(lb, w.S_max))
    assert torch.equal(lens.long(), expect)
    for b in range(1, w.B):
        p = int(lb[b])
        assert torch.equal(kc[b, :, p].view(torch.int16), kn[b, 0].view(torch.int16))
        assert torch.equal(vc[b, :, p].view(torch.int16), vn[b, 0].view(torch.int16))
    # rows other than the appended ones are unchanged
    mask = torch.ones(kc.shape[:3], dtype=torch.bool, device=DEV)
    for b in range(1, w.B):
        mask[b, :, int(lb[b])] = False
    assert torch.equal(kc[mask].view(torch.int16), k_before[mask].view(torch.int16))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("h_q,g", [(16, 1), (64, 2), (128, 1), (32, 2)])
def test_decode_large_groups_tensor_core_path(d, h_q, g):
    """Groups of 16..128 query heads (stacked 32 rows per work item, larger
    groups in several items): ragged lengths including 0, 1 and stage
    boundaries, garbage past the lengths."""
    B, S = 6, 4500
    q = rand_bf16((B, h_q, d), 81 + h_q)
    kc = rand_bf16((B, g, S, d), 82 + h_q)
    vc = rand_bf16((B, g, S, d), 83 + h_q)
    lens_l = [4500, 0, 1, 63, 65, 2049]
    lens = torch.tensor(lens_l, dtype=torch.int32, device=DEV)
    o_clean, lse_clean = run_decode(q, kc, vc, lens, 1.0 / math.sqrt(d))
    for b, n in enumerate(lens_l):
        kc[b, :, n:] = float("nan")
        vc[b, :, n:] = float("inf")
    o, lse = run_decode(q, kc, vc, lens, 1.0 / math.sqrt(d))
    assert torch.equal(o, o_clean) and torch.equal(lse, lse_clean)
    assert torch.all(o[1] == 0) and torch.all(torch.isneginf(lse[1]))
    o_ref, lse_ref = oracle.decode(f64(q), f64(kc), f64(vc), lens_l, 1.0 / math.sqrt(d))
    assert_close(f64(o), o_ref, f"decode G={h_q // g} d={d}")
    keep = [b for b, n in enumerate(lens_l) if n > 0]  # the empty row's lse is -inf (checked above)
    assert_close(f64(lse)[keep], lse_ref[keep], f"decode lse G={h_q // g} d={d}")
    o16, _ = run_decode(q, kc, vc, lens, 1.0 / math.sqrt(d), out_dtype=torch.bfloat16)
    assert_close(f64(o16), o_ref, "bf16 out")
