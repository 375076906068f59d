"""GPU parity of the score-bias variants and the chunked prefill over a cache.

Sliding window and ALiBi (the variants the pages name) on prefill and
decode, and the chunked prefill in which T new tokens attend to a
[B, g, S_max, d] KV cache, all through the C interface against the fp64
oracle on the same seeded bf16 inputs. Tolerance as in the other parity
tests: max abs error <= 1e-2, mean abs error <= 1e-3, for O and for lse.
Output and lse buffers sit between NaN guard bands that must stay untouched.
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
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: non-finite entries differ"
    err = np.abs(got[fin] - ref[fin])
    assert err.max() <= max_abs, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= mean_abs, f"{what}: mean abs err {err.mean():.3e}"


def rand_bf16(shape, seed):
    return inputs.random_bf16(shape, seed, device="cpu").to(DEV)


def alibi_slopes(h_q):
    # the usual geometric slopes 2^(-8 h / h_q), h = 1 .. h_q
    return torch.tensor([2.0 ** (-8.0 * (h + 1) / h_q) for h in range(h_q)],
                        dtype=torch.float32, device=DEV)


# ---------------------------------------------------------------------------
# prefill: sliding window and ALiBi
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("L,window", [(200, 1), (384, 100), (300, 128), (257, 129),
                                      (1000, 256), (129, 500)])
def test_prefill_sliding_window(d, L, window):
    B, h_q, g = 2, 8, 2
    q = rand_bf16((B, L, h_q, d), 300 + L)
    k = rand_bf16((B, L, g, d), 301 + L)
    v = rand_bf16((B, L, g, d), 302 + L)
    scale = 1.0 / math.sqrt(d)
    go = guard.empty((B, L, h_q, d), torch.float32, DEV)
    gl = guard.empty((B, h_q, L), torch.float32, DEV)
    lse = gl.tensor
    o = gqa.gqa_prefill_fwd(q, k, v, causal=True, scale=scale, window=window, lse=lse,
                            out=go.tensor)
    torch.cuda.synchronize()
    go.assert_bands(f"windowed prefill O L={L}")
    gl.assert_bands(f"windowed prefill lse L={L}")
    o_ref, lse_ref = oracle.prefill(f64(q), f64(k), f64(v), True, scale, window=window)
    assert_close(f64(o), o_ref, f"window {window} L={L} d={d}")
    assert_close(f64(lse), lse_ref, "lse")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("h_q,g", [(8, 2), (32, 8), (16, 16)])
def test_prefill_alibi(d, causal, h_q, g):
    B, L = 2, 300
    q = rand_bf16((B, L, h_q, d), 400 + h_q + g)
    k = rand_bf16((B, L, g, d), 401 + h_q + g)
    v = rand_bf16((B, L, g, d), 402 + h_q + g)
    scale = 1.0 / math.sqrt(d)
    slopes = alibi_slopes(h_q)
    go = guard.empty((B, L, h_q, d), torch.float32, DEV)
    gl = guard.empty((B, h_q, L), torch.float32, DEV)
    lse = gl.tensor
    o = gqa.gqa_prefill_fwd(q, k, v, causal=causal, scale=scale, alibi_slopes=slopes, lse=lse,
                            out=go.tensor)
    torch.cuda.synchronize()
    go.assert_bands("ALiBi prefill O")
    gl.assert_bands("ALiBi prefill lse")
    o_ref, lse_ref = oracle.prefill(f64(q), f64(k), f64(v), causal, scale,
                                    alibi_slopes=slopes.cpu().numpy().astype(np.float64))
    assert_close(f64(o), o_ref, f"alibi causal={causal} h_q={h_q} g={g}")
    assert_close(f64(lse), lse_ref, "lse")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("window", [0, 200])
def test_prefill_alibi_window_bf16_output(d, window):
    # the variant instantiations through the bf16-output epilogue, guarded
    B, L, h_q, g = 2, 300, 16, 4
    q = rand_bf16((B, L, h_q, d), 450 + window + d)
    k = rand_bf16((B, L, g, d), 451 + window + d)
    v = rand_bf16((B, L, g, d), 452 + window + d)
    scale = 1.0 / math.sqrt(d)
    slopes = alibi_slopes(h_q)
    go = guard.empty((B, L, h_q, d), torch.bfloat16, DEV)
    o = gqa.gqa_prefill_fwd(q, k, v, causal=True, scale=scale, window=window,
                            alibi_slopes=slopes, out=go.tensor)
    torch.cuda.synchronize()
    go.assert_bands("ALiBi/window prefill bf16 O")
    o_ref, _ = oracle.prefill(f64(q), f64(k), f64(v), True, scale, window=window,
                              alibi_slopes=slopes.cpu().numpy().astype(np.float64))
    assert_close(f64(o), o_ref, f"alibi window={window} d={d} bf16 output")


def test_prefill_window_and_alibi_llama_shape_sampled_rows():
    B, L, h_q, g, d, W = 2, 2048, 32, 8, 128, 512
    q = rand_bf16((B, L, h_q, d), 501)
    k = rand_bf16((B, L, g, d), 502)
    v = rand_bf16((B, L, g, d), 503)
    scale = 1.0 / math.sqrt(d)
    slopes = alibi_slopes(h_q)
    o = gqa.gqa_prefill_fwd(q, k, v, causal=True, scale=scale, window=W, alibi_slopes=slopes)
    torch.cuda.synchronize()
    sl = slopes.cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(7)
    for b, pos in [(0, 0), (1, L - 1), (0, W - 1), (1, W)] + [
            (int(rng.integers(B)), int(rng.integers(L))) for _ in range(8)]:
        lo = max(0, pos - W + 1)
        o_r, _ = oracle.prefill(f64(q[b:b + 1, pos:pos + 1]), f64(k[b:b + 1, lo:pos + 1]),
                                f64(v[b:b + 1, lo:pos + 1]), True, scale, q_offset=pos - lo,
                                alibi_slopes=sl)
        assert_close(f64(o[b, pos]), o_r[0, 0], f"row {pos} of batch {b}")


def test_prefill_window_wider_than_sequence_equals_plain_causal():
    B, L, h_q, g, d = 1, 333, 8, 4, 64
    q, k, v = rand_bf16((B, L, h_q, d), 511), rand_bf16((B, L, g, d), 512), rand_bf16(
        (B, L, g, d), 513)
    a = gqa.gqa_prefill_fwd(q, k, v, causal=True, window=L)
    b = gqa.gqa_prefill_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


# ---------------------------------------------------------------------------
# chunked prefill over the KV cache
# ---------------------------------------------------------------------------

def _cached_case(B, T, h_q, g, d, S_max, lens, seed, window=0, alibi=False, nan_tail=True,
                 out_dtype=torch.float32):
    kc = rand_bf16((B, g, S_max, d), seed)
    vc = rand_bf16((B, g, S_max, d), seed + 1)
    q = rand_bf16((B, T, h_q, d), seed + 2)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=DEV)
    if nan_tail:
        for b, n in enumerate(lens):
            kc[b, :, n:] = float("nan")
            vc[b, :, n:] = float("nan")
    slopes = alibi_slopes(h_q) if alibi else None
    scale = 1.0 / math.sqrt(d)
    go = guard.empty((B, T, h_q, d), out_dtype, DEV)
    gl = guard.empty((B, h_q, T), torch.float32, DEV)
    lse = gl.tensor
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = gqa.gqa_prefill_kvcache_fwd(q, kc, vc, lens_t, scale=scale, lse=lse, window=window,
                                    alibi_slopes=slopes, status=status, out=go.tensor)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    go.assert_bands(f"chunked prefill O T={T}")
    gl.assert_bands(f"chunked prefill lse T={T}")
    sl = None if slopes is None else slopes.cpu().numpy().astype(np.float64)
    kc64 = np.nan_to_num(f64(kc))  # rows past the length are never visible to the oracle
    vc64 = np.nan_to_num(f64(vc))
    o_ref, lse_ref = oracle.prefill_cached(f64(q), kc64, vc64, lens, scale, window=window,
                                           alibi_slopes=sl)
    return o, lse, o_ref, lse_ref


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("T,lens", [(1, [1, 700, 1024]), (7, [7, 130, 999]),
                                    (64, [64, 600, 1000]), (129, [129, 300, 1024]),
                                    (300, [1024, 300, 777])])
def test_prefill_kvcache_ragged(d, T, lens):
    o, lse, o_ref, lse_ref = _cached_case(3, T, 32, 8, d, 1024, lens, seed=600 + T + d)
    assert_close(f64(o), o_ref, f"kvcache T={T} d={d}")
    assert_close(f64(lse), lse_ref, "lse")


@pytest.mark.parametrize("h_q,g", [(8, 8), (32, 1), (16, 4)])
@pytest.mark.parametrize("window,alibi", [(0, True), (96, False), (200, True)])
def test_prefill_kvcache_variants(h_q, g, window, alibi):
    o, lse, o_ref, lse_ref = _cached_case(2, 100, h_q, g, 128, 900, [900, 333], seed=700 + h_q,
                                          window=window, alibi=alibi)
    assert_close(f64(o), o_ref, f"kvcache window={window} alibi={alibi}")
    assert_close(f64(lse), lse_ref, "lse")


@pytest.mark.parametrize("d", [64, 128])
def test_prefill_kvcache_bf16_output(d):
    o, lse, o_ref, lse_ref = _cached_case(3, 129, 32, 8, d, 1024, [129, 600, 1024], seed=750 + d,
                                          out_dtype=torch.bfloat16)
    assert o.dtype == torch.bfloat16
    assert_close(f64(o), o_ref, f"kvcache bf16 output d={d}")
    assert_close(f64(lse), lse_ref, "lse")


def test_append_then_chunked_prefill_then_decode_pipeline():
    """Prompt prefill, a chunk appended and prefilled against the cache, then
    a decode token: the path a serving loop runs, each step against the oracle."""
    B, h_q, g, d, S_max, P, T = 2, 32, 8, 128, 512, 200, 48
    kc = torch.zeros((B, g, S_max, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    lens = torch.zeros((B,), dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    k_all = rand_bf16((B, P + T + 1, g, d), 801)
    v_all = rand_bf16((B, P + T + 1, g, d), 802)
    q_all = rand_bf16((B, P + T + 1, h_q, d), 803)
    gqa.kv_cache_append(kc, vc, lens, k_all[:, :P].contiguous(), v_all[:, :P].contiguous(),
                        status=status)
    gqa.kv_cache_append(kc, vc, lens, k_all[:, P:P + T].contiguous(),
                        v_all[:, P:P + T].contiguous(), status=status)
    o_chunk = gqa.gqa_prefill_kvcache_fwd(q_all[:, P:P + T].contiguous(), kc, vc, lens)
    gqa.kv_cache_append(kc, vc, lens, k_all[:, P + T:].contiguous(), v_all[:, P + T:].contiguous(),
                        status=status)
    o_dec = gqa.gqa_decode_fwd(q_all[:, P + T].contiguous(), kc, vc, lens)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_full, _ = oracle.prefill(f64(q_all), f64(k_all), f64(v_all), True, 1.0 / math.sqrt(d))
    assert_close(f64(o_chunk), o_full[:, P:P + T], "chunk rows")
    assert_close(f64(o_dec), o_full[:, P + T], "decode row")


def test_kvcache_bad_length_is_flagged():
    B, T, h_q, g, d, S_max = 2, 16, 8, 2, 64, 256
    kc = rand_bf16((B, g, S_max, d), 901)
    vc = rand_bf16((B, g, S_max, d), 902)
    q = rand_bf16((B, T, h_q, d), 903)
    lens = torch.tensor([8, 100], dtype=torch.int32, device=DEV)  # 8 < T
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gqa.gqa_prefill_kvcache_fwd(q, kc, vc, lens, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == gqa.GQA_ERR_BAD_LENGTH


# ---------------------------------------------------------------------------
# decode: sliding window and ALiBi
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("G_cfg", [(32, 8), (32, 1), (8, 8)])
@pytest.mark.parametrize("window,alibi", [(1, False), (300, False), (0, True), (1000, True)])
def test_decode_window_alibi(G_cfg, window, alibi):
    h_q, g = G_cfg
    B, d, S_max = 4, 128, 3000
    kc = rand_bf16((B, g, S_max, d), 1000 + window)
    vc = rand_bf16((B, g, S_max, d), 1001 + window)
    q = rand_bf16((B, h_q, d), 1002 + window)
    lens_l = [3000, 1, 299, 1777]
    lens = torch.tensor(lens_l, dtype=torch.int32, device=DEV)
    if window > 0:
        # rows before the window must never be read
        for b, n in enumerate(lens_l):
            lo = max(0, n - window)
            kc[b, :, :lo] = float("nan")
            vc[b, :, :lo] = float("nan")
    slopes = alibi_slopes(h_q) if alibi else None
    gl = guard.empty((B, h_q), torch.float32, DEV)
    go = guard.empty((B, h_q, d), torch.float32, DEV)
    lse = gl.tensor
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = gqa.gqa_decode_fwd(q, kc, vc, lens, scale=0.0884, lse=lse, window=window,
                           alibi_slopes=slopes, status=status, out=go.tensor)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    go.assert_bands("windowed decode O")
    gl.assert_bands("windowed decode lse")
    sl = None if slopes is None else slopes.cpu().numpy().astype(np.float64)
    o_ref, lse_ref = oracle.decode(f64(q), np.nan_to_num(f64(kc)), np.nan_to_num(f64(vc)),
                                   lens_l, 0.0884, window=window, alibi_slopes=sl)
    assert_close(f64(o), o_ref, f"decode window={window} alibi={alibi}")
    assert_close(f64(lse), lse_ref, "lse")


@pytest.mark.parametrize("alibi", [False, True])
def test_decode_window_split_from_the_window(alibi):
    # 30 sequences x 8 K/V heads fill the CTA slots with one split per
    # segment, so a 256-row window is read as one item per segment while the
    # 4096-row cache (more than one longest item) is split in two. Rows before
    # the window hold NaN and must never be read.
    B, h_q, g, d, S_max, W = 30, 32, 8, 64, 4096, 256
    kc = rand_bf16((B, g, S_max, d), 1201)
    vc = rand_bf16((B, g, S_max, d), 1202)
    q = rand_bf16((B, h_q, d), 1203)
    gen = torch.Generator().manual_seed(1204)
    lens_l = torch.randint(2100, S_max + 1, (B,), generator=gen).tolist()
    lens_l[0], lens_l[1] = S_max, W - 3  # a full cache and one shorter than the window
    for b, n in enumerate(lens_l):
        lo = max(0, n - W)
        kc[b, :, :lo] = float("nan")
        vc[b, :, :lo] = float("nan")
    slopes = alibi_slopes(h_q) if alibi else None
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    go = guard.empty((B, h_q, d), torch.float32, DEV)
    o = gqa.gqa_decode_fwd(q, kc, vc, torch.tensor(lens_l, dtype=torch.int32, device=DEV),
                           scale=0.125, window=W, alibi_slopes=slopes, status=status,
                           out=go.tensor)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    go.assert_bands("window-split decode O")
    # the oracle reads only the window: its rows moved to the front of a
    # compact cache (ALiBi depends on relative positions only)
    n_w = [min(W, n) for n in lens_l]
    kw = np.zeros((B, g, W, d))
    vw = np.zeros((B, g, W, d))
    for b, n in enumerate(lens_l):
        kw[b, :, :n_w[b]] = f64(kc[b, :, n - n_w[b]:n])
        vw[b, :, :n_w[b]] = f64(vc[b, :, n - n_w[b]:n])
    sl = None if slopes is None else slopes.cpu().numpy().astype(np.float64)
    o_ref, _ = oracle.decode(f64(q), kw, vw, n_w, 0.125, alibi_slopes=sl)
    assert_close(f64(o), o_ref, f"window-split decode alibi={alibi}")


def test_decode_window_longer_than_the_cache_with_few_segments():
    # 4 segments and a window longer than the cache: splitting W' + 63 rows
    # by the cache rule would need more splits than the workspace holds, so
    # the window's rows are spread over the workspace's splits
    h_q, g = 32, 1
    B, d, S_max = 4, 128, 3000
    kc = rand_bf16((B, g, S_max, d), 1301)
    vc = rand_bf16((B, g, S_max, d), 1302)
    q = rand_bf16((B, h_q, d), 1303)
    lens_l = [3000, 2999, 64, 1]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = gqa.gqa_decode_fwd(q, kc, vc, torch.tensor(lens_l, dtype=torch.int32, device=DEV),
                           scale=0.0884, window=5000, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    o_ref, _ = oracle.decode(f64(q), f64(kc), f64(vc), lens_l, 0.0884)
    assert_close(f64(o), o_ref, "window > cache, few segments")


@pytest.mark.parametrize("window", [0, 300])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B,h_q,g,d,S_max", [(40, 32, 8, 128, 1500), (240, 32, 1, 128, 256),
                                             (40, 8, 8, 64, 700)])
def test_decode_single_split_writes_the_output(window, out_dtype, B, h_q, g, d, S_max):
    # enough (sequence, K/V head) segments to fill the CTA slots with one split
    # each and a cache that fits one split: the split pass merges its consumer
    # warps' partials and writes O and lse itself (no combine pass). Empty
    # sequences, one-row and full ones, NaN rows past the lengths.
    kc = rand_bf16((B, g, S_max, d), 1400 + B + g)
    vc = rand_bf16((B, g, S_max, d), 1401 + B + g)
    q = rand_bf16((B, h_q, d), 1402 + B + g)
    gen = torch.Generator().manual_seed(1403 + B)
    lens_l = torch.randint(0, S_max + 1, (B,), generator=gen).tolist()
    lens_l[:5] = [0, 1, S_max, 63, 65 if S_max > 65 else S_max]
    for b, n in enumerate(lens_l):
        kc[b, :, n:] = float("nan")
        vc[b, :, n:] = float("nan")
    go = guard.empty((B, h_q, d), out_dtype, DEV)
    gl = guard.empty((B, h_q), torch.float32, DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gqa.gqa_decode_fwd(q, kc, vc, torch.tensor(lens_l, dtype=torch.int32, device=DEV),
                       scale=0.1, window=window, lse=gl.tensor, out=go.tensor, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    go.assert_bands("single-split decode O")
    gl.assert_bands("single-split decode lse")
    o_ref, lse_ref = oracle.decode(f64(q), np.nan_to_num(f64(kc)), np.nan_to_num(f64(vc)),
                                   lens_l, 0.1, window=window)
    assert_close(f64(go.tensor), o_ref, f"single-split decode B={B} g={g} window={window}")
    assert_close(f64(gl.tensor), lse_ref, "single-split decode lse")


def test_decode_single_split_flags_a_bad_length():
    B, h_q, g, d, S_max = 40, 32, 8, 128, 1000
    kc = rand_bf16((B, g, S_max, d), 1501)
    vc = rand_bf16((B, g, S_max, d), 1502)
    q = rand_bf16((B, h_q, d), 1503)
    lens = torch.full((B,), 500, dtype=torch.int32, device=DEV)
    lens[7] = -3
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gqa.gqa_decode_fwd(q, kc, vc, lens, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == gqa.GQA_ERR_BAD_LENGTH


def test_decode_equals_one_token_chunked_prefill_with_bias():
    B, h_q, g, d, S_max = 3, 32, 8, 128, 1500
    kc = rand_bf16((B, g, S_max, d), 1101)
    vc = rand_bf16((B, g, S_max, d), 1102)
    q = rand_bf16((B, h_q, d), 1103)
    lens = torch.tensor([1500, 17, 640], dtype=torch.int32, device=DEV)
    slopes = alibi_slopes(h_q)
    o_d = gqa.gqa_decode_fwd(q, kc, vc, lens, window=400, alibi_slopes=slopes)
    o_p = gqa.gqa_prefill_kvcache_fwd(q[:, None].contiguous(), kc, vc, lens, window=400,
                                      alibi_slopes=slopes)
    torch.cuda.synchronize()
    assert_close(f64(o_d), f64(o_p[:, 0]), "decode vs one-token chunk", max_abs=5e-3)
