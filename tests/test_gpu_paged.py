"""GPU parity of the paged KV cache (group-aligned pages, block table).

Paged decode and paged append through the C interface against the fp64
oracle's paged functions (which are pinned to the contiguous ones), on
shuffled physical pages, ragged lengths, page sizes below and above the
64-token decode stage, and with the window / ALiBi options. Outputs and page
pools sit between NaN guard bands that every call must leave untouched.
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
    assert got.shape == ref.shape
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: non-finite entries differ"
    err = np.abs(got[fin] - ref[fin])
    assert err.max() <= max_abs, f"{what}: max abs err {err.max():.3e}"
    assert err.mean() <= mean_abs, f"{what}: mean abs err {err.mean():.3e}"


def paged_case(B, h_q, g, d, page, max_blocks, lens, seed, spare=3):
    """Pool with shuffled pages; unused table entries point at -1 (never read)."""
    need = [(n + page - 1) // page for n in lens]
    num_pages = sum(need) + spare
    rng = np.random.default_rng(seed)
    perm = rng.permutation(num_pages)
    table = np.full((B, max_blocks), -1, dtype=np.int32)
    k = 0
    for b in range(B):
        for i in range(need[b]):
            table[b, i] = perm[k]
            k += 1
    kp = inputs.random_bf16((num_pages, g, page, d), seed, device="cpu").to(DEV)
    vp = inputs.random_bf16((num_pages, g, page, d), seed + 1, device="cpu").to(DEV)
    q = inputs.random_bf16((B, h_q, d), seed + 2, device="cpu").to(DEV)
    return q, kp, vp, torch.from_numpy(table).to(DEV), table


@pytest.mark.parametrize("page", [16, 32, 64, 128, 256])
@pytest.mark.parametrize("h_q,g,d", [(32, 8, 128), (8, 2, 64), (32, 1, 128)])
def test_paged_decode_matches_oracle(page, h_q, g, d):
    B, max_blocks = 4, 2048 // page
    lens = [2048, 1, 777, 1500]
    q, kp, vp, table_t, table = paged_case(B, h_q, g, d, page, max_blocks, lens, 11 + page + g)
    lens_t = torch.tensor(lens, dtype=torch.int32, device=DEV)
    gl = guard.empty((B, h_q), torch.float32, DEV)
    go = guard.empty((B, h_q, d), torch.float32, DEV)
    lse = gl.tensor
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = gqa.gqa_decode_paged_fwd(q, kp, vp, table_t, lens_t, lse=lse, status=status,
                                 out=go.tensor)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    go.assert_bands(f"paged decode O page={page}")
    gl.assert_bands(f"paged decode lse page={page}")
    scale = 1.0 / math.sqrt(d)
    o_ref, lse_ref = oracle.decode_paged(f64(q), f64(kp), f64(vp), table, lens, page, scale)
    assert_close(f64(o), o_ref, f"paged decode page={page}")
    assert_close(f64(lse), lse_ref, "lse")


@pytest.mark.parametrize("page", [16, 32, 128])
@pytest.mark.parametrize("window,alibi", [(100, False), (0, True), (700, True), (1, False)])
def test_paged_decode_window_alibi(window, alibi, page):
    B, h_q, g, d = 3, 32, 8, 128
    max_blocks = 1280 // page
    lens = [1280, 45, 999]
    q, kp, vp, table_t, table = paged_case(B, h_q, g, d, page, max_blocks, lens, 77)
    if window > 0:
        # pages wholly before the window may already be released by the caller
        for b, n in enumerate(lens):
            table_t[b, : max(0, n - window) // page] = -1
    lens_t = torch.tensor(lens, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    slopes = torch.tensor([2.0 ** (-8.0 * (h + 1) / h_q) for h in range(h_q)],
                          dtype=torch.float32, device=DEV) if alibi else None
    o = gqa.gqa_decode_paged_fwd(q, kp, vp, table_t, lens_t, window=window, alibi_slopes=slopes,
                                 status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sl = None if slopes is None else slopes.cpu().numpy().astype(np.float64)
    o_ref, _ = oracle.decode_paged(f64(q), f64(kp), f64(vp), table, lens, page,
                                   1.0 / math.sqrt(d), window=window, alibi_slopes=sl)
    assert_close(f64(o), o_ref, f"paged decode window={window} alibi={alibi}")


def test_paged_decode_equals_contiguous_decode():
    """Pages in identity order are a reshaped contiguous cache: both paths agree."""
    B, h_q, g, d, S, page = 2, 32, 8, 128, 1024, 64
    kc = inputs.random_bf16((B, g, S, d), 91, device="cpu").to(DEV)
    vc = inputs.random_bf16((B, g, S, d), 92, device="cpu").to(DEV)
    q = inputs.random_bf16((B, h_q, d), 93, device="cpu").to(DEV)
    lens = torch.tensor([1000, 333], dtype=torch.int32, device=DEV)
    nb = S // page
    to_pool = lambda c: c.view(B, g, nb, page, d).permute(0, 2, 1, 3, 4).reshape(
        B * nb, g, page, d).contiguous()
    table = torch.arange(B * nb, dtype=torch.int32, device=DEV).view(B, nb).contiguous()
    o_p = gqa.gqa_decode_paged_fwd(q, to_pool(kc), to_pool(vc), table, lens)
    o_c = gqa.gqa_decode_fwd(q, kc, vc, lens)
    torch.cuda.synchronize()
    assert_close(f64(o_p), f64(o_c), "paged vs contiguous", max_abs=1e-5, mean_abs=1e-6)


@pytest.mark.parametrize("page", [16, 64, 128])
def test_paged_append_bit_exact_then_decode(page):
    B, h_q, g, d, max_blocks, T = 3, 16, 4, 128, 8, 20
    cap = page * max_blocks
    lens0 = [0, page - 3, cap - 5]  # the last one overflows its capacity
    q, kp, vp, table_t, table = paged_case(B, h_q, g, d, page, max_blocks,
                                           [cap] * B, 300 + page)
    kn = inputs.random_bf16((B, T, g, d), 301, device="cpu").to(DEV)
    vn = inputs.random_bf16((B, T, g, d), 302, device="cpu").to(DEV)
    lens = torch.tensor(lens0, dtype=torch.int32, device=DEV)
    bits = lambda t: t.view(torch.int16).cpu().numpy()
    k_ref, v_ref, lens_ref, st_ref = oracle.append_paged(bits(kp), bits(vp), table, lens0,
                                                         bits(kn), bits(vn), page)
    gk, gv = guard.copy_of(kp), guard.copy_of(vp)
    kp, vp = gk.tensor, gv.tensor
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gqa.kv_cache_append_paged(kp, vp, table_t, lens, kn, vn, status=status)
    torch.cuda.synchronize()
    gk.assert_bands(f"paged append K pool page={page}")
    gv.assert_bands(f"paged append V pool page={page}")
    assert np.array_equal(bits(kp), k_ref) and np.array_equal(bits(vp), v_ref)
    assert list(lens.cpu().numpy()) == list(lens_ref)
    assert int(status.item()) == st_ref == oracle.APPEND_CACHE_FULL
    o = gqa.gqa_decode_paged_fwd(q, kp, vp, table_t, lens)
    torch.cuda.synchronize()
    o_ref, _ = oracle.decode_paged(f64(q), oracle.bf16_bits_to_f64(k_ref.view(np.uint16)),
                                   oracle.bf16_bits_to_f64(v_ref.view(np.uint16)), table,
                                   lens_ref, page, 1.0 / math.sqrt(d))
    assert_close(f64(o), o_ref, "decode after paged append")


def test_paged_bad_table_entry_is_flagged_not_faulting():
    B, h_q, g, d, page, max_blocks = 2, 8, 2, 64, 64, 4
    q, kp, vp, table_t, table = paged_case(B, h_q, g, d, page, max_blocks, [256, 100], 55)
    table_t[1, 0] = 10_000  # past the pool
    lens = torch.tensor([256, 100], dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = gqa.gqa_decode_paged_fwd(q, kp, vp, table_t, lens, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == gqa.GQA_ERR_BAD_PAGE
    # the sequence with valid pages is unaffected
    o_ref, _ = oracle.decode_paged(f64(q[:1]), f64(kp), f64(vp), table[:1], [256], page,
                                   1.0 / math.sqrt(d))
    assert_close(f64(o[:1]), o_ref, "valid sequence next to a bad one")
