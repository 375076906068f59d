"""Pins of the CPU oracle to facts other than itself (no GPU needed).

Each check ties the oracle to something independent of its own code:
PyTorch's library attention (``scaled_dot_product_attention`` with
``enable_gqa``) in fp64, brute-force loops on tiny inputs, the MHA and MQA
special cases written in their own forms, hand-derived closed-form fixtures
(tests/golden/closed_form_gqa.json) and invariants of the definition. The
mutation tests at the end plant plausible mistakes in the oracle and check
that at least one pin catches each of them.
"""

import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import gqa_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_gqa.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa(q, k, v, causal, scale):
    """PyTorch library attention in fp64; inputs in the [B, L, heads, d] layout."""
    tq = torch.from_numpy(q).transpose(1, 2)
    tk = torch.from_numpy(k).transpose(1, 2)
    tv = torch.from_numpy(v).transpose(1, 2)
    o = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale,
                                       enable_gqa=True)
    return o.transpose(1, 2).numpy()


# ---------------------------------------------------------------------------
# Pin checks (raise AssertionError on failure); reused by the mutation tests.
# ---------------------------------------------------------------------------

def check_golden_prefill():
    c = _golden()["prefill_mqa_L2"]
    q, k, v = (np.array(c[n], dtype=np.float64) for n in ("q", "k", "v"))
    o, lse = oracle.prefill(q, k, v, causal=False, scale=c["scale"])
    np.testing.assert_allclose(o, c["o_noncausal"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, c["lse_noncausal"], rtol=0, atol=1e-12)
    o, lse = oracle.prefill(q, k, v, causal=True, scale=c["scale"])
    np.testing.assert_allclose(o, c["o_causal"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, c["lse_causal"], rtol=0, atol=1e-12)


def check_golden_decode():
    c = _golden()["decode_head_map"]
    o, lse = oracle.decode(np.array(c["q"]), np.array(c["k_cache"]),
                           np.array(c["v_cache"]), np.array(c["seq_lens"]),
                           scale=c["scale"])
    np.testing.assert_allclose(o, c["o"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, c["lse"], rtol=0, atol=1e-12)


def check_against_sdpa():
    for (B, L, h_q, g, d, causal, seed) in [
        (2, 7, 8, 2, 16, True, 1), (1, 9, 8, 4, 8, False, 2),
        (2, 5, 4, 4, 8, True, 3), (1, 6, 6, 1, 4, False, 4),
        (1, 13, 32, 8, 16, True, 5), (3, 4, 2, 1, 8, True, 6),
    ]:
        q = _rand((B, L, h_q, d), seed)
        k = _rand((B, L, g, d), seed + 100)
        v = _rand((B, L, g, d), seed + 200)
        scale = 1.0 / math.sqrt(d)
        o, _ = oracle.prefill(q, k, v, causal, scale)
        np.testing.assert_allclose(o, _sdpa(q, k, v, causal, scale), rtol=0, atol=1e-12)


def check_permutation_within_group():
    B, L, h_q, g, d = 1, 6, 8, 2, 8
    G = h_q // g
    q = _rand((B, L, h_q, d), 11)
    k = _rand((B, L, g, d), 12)
    v = _rand((B, L, g, d), 13)
    o, _ = oracle.prefill(q, k, v, True, 0.3)
    # permute query heads inside each group: outputs permute the same way
    perm = np.concatenate([np.random.default_rng(14).permutation(G) + j * G
                           for j in range(g)])
    o_p, _ = oracle.prefill(q[:, :, perm, :], k, v, True, 0.3)
    np.testing.assert_allclose(o_p, o[:, :, perm, :], rtol=0, atol=1e-12)
    # move a head to the other group: its output must change
    swap = np.arange(h_q)
    swap[0], swap[G] = G, 0
    o_s, _ = oracle.prefill(q[:, :, swap, :], k, v, True, 0.3)
    assert np.max(np.abs(o_s[:, :, 0, :] - o[:, :, G, :])) > 1e-3


def check_rows_sum_to_one():
    q = _rand((2, 5, 4, 8), 21)
    k = _rand((2, 5, 2, 8), 22)
    for causal in (False, True):
        p = oracle.attention_probs(q, k, causal, 0.5)
        np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-12)
        assert np.all(p >= 0)
        if causal:
            iu = np.triu_indices(5, 1)
            assert np.all(p[:, :, iu[0], iu[1]] == 0.0)


def check_causal_row0_is_v0():
    q = _rand((2, 4, 8, 8), 31)
    k = _rand((2, 4, 2, 8), 32)
    v = _rand((2, 4, 2, 8), 33)
    o, _ = oracle.prefill(q, k, v, True, 0.25)
    for h in range(8):
        assert np.array_equal(o[:, 0, h, :], v[:, 0, h // 4, :])


def _band_mask(Lq, Lk, q_offset, window):
    """Boolean visibility built with torch primitives (True = visible)."""
    i = torch.arange(Lq)[:, None] + q_offset
    j = torch.arange(Lk)[None, :]
    vis = j <= i
    if window > 0:
        vis = vis & (j > i - window)
    return vis


def check_window_against_sdpa_mask():
    for (B, L, h_q, g, d, W, seed) in [(2, 11, 8, 2, 8, 3, 41), (1, 9, 4, 4, 16, 1, 42),
                                       (1, 12, 8, 1, 8, 5, 43)]:
        q = _rand((B, L, h_q, d), seed)
        k = _rand((B, L, g, d), seed + 1)
        v = _rand((B, L, g, d), seed + 2)
        scale = 1.0 / math.sqrt(d)
        o, _ = oracle.prefill(q, k, v, True, scale, window=W)
        tq, tk, tv = (torch.from_numpy(x).transpose(1, 2) for x in (q, k, v))
        ref = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=_band_mask(L, L, 0, W),
                                             scale=scale, enable_gqa=True)
        np.testing.assert_allclose(o, ref.transpose(1, 2).numpy(), rtol=0, atol=1e-12)


def check_window_one_returns_own_v():
    q = _rand((2, 6, 8, 8), 51)
    k = _rand((2, 6, 2, 8), 52)
    v = _rand((2, 6, 2, 8), 53)
    o, _ = oracle.prefill(q, k, v, True, 0.4, window=1)
    for h in range(8):
        assert np.array_equal(o[:, :, h, :], v[:, :, h // 4, :])


def check_alibi_causal_against_sdpa_augmented():
    # causal ALiBi: -slope*(i - j) = slope*j - slope*i, and the per-row term
    # cancels in the softmax; so it equals plain attention on per-head
    # vectors augmented with one coordinate: q' = [q, 1], k'_j = [k_j, slope*j/scale]
    B, L, h_q, g, d = 2, 10, 8, 2, 8
    q = _rand((B, L, h_q, d), 61)
    k = _rand((B, L, g, d), 62)
    v = _rand((B, L, g, d), 63)
    slopes = np.array([2.0 ** (-8.0 * (h + 1) / h_q) for h in range(h_q)])
    scale = 1.0 / math.sqrt(d)
    o, _ = oracle.prefill(q, k, v, True, scale, alibi_slopes=slopes)
    G = h_q // g
    tq = torch.from_numpy(q).transpose(1, 2)                       # [B, h_q, L, d]
    tk = torch.from_numpy(k).transpose(1, 2).repeat_interleave(G, dim=1)
    tv = torch.from_numpy(v).transpose(1, 2).repeat_interleave(G, dim=1)
    pos = torch.arange(L, dtype=torch.float64)
    extra_k = torch.from_numpy(slopes)[:, None] * pos[None, :] / scale  # [h_q, L]
    qa = torch.cat([tq, torch.ones(B, h_q, L, 1, dtype=torch.float64)], dim=-1)
    ka = torch.cat([tk, extra_k[None, :, :, None].expand(B, h_q, L, 1)], dim=-1)
    ref = F.scaled_dot_product_attention(qa, ka, tv, is_causal=True, scale=scale)
    np.testing.assert_allclose(o, ref.transpose(1, 2).numpy(), rtol=0, atol=1e-10)


def _all_checks():
    return [check_golden_prefill, check_golden_decode, check_against_sdpa,
            check_permutation_within_group, check_rows_sum_to_one,
            check_causal_row0_is_v0, check_window_against_sdpa_mask,
            check_window_one_returns_own_v, check_alibi_causal_against_sdpa_augmented]


# ---------------------------------------------------------------------------
# The pins themselves
# ---------------------------------------------------------------------------

def test_golden_prefill_closed_form():
    check_golden_prefill()


def test_golden_decode_head_map_closed_form():
    check_golden_decode()


def test_golden_append_closed_form():
    c = _golden()["append_overflow"]
    B, g, S, d = c["B"], c["g"], c["S_max"], c["d"]
    kc = -np.ones((B, g, S, d))
    vc = -np.ones((B, g, S, d))
    kc2, vc2, lens2, status = oracle.append(kc, vc, np.array(c["seq_lens"]),
                                            np.array(c["k_new"]), np.array(c["v_new"]))
    assert np.array_equal(kc2, np.array(c["k_cache_after"]))
    assert np.array_equal(vc2, np.array(c["v_cache_after"]))
    assert list(lens2) == c["seq_lens_after"]
    assert status == c["status"] == oracle.APPEND_CACHE_FULL


def test_prefill_matches_library_sdpa_fp64():
    check_against_sdpa()


def test_prefill_brute_force_loops_tiny():
    """Per-element loops over an explicitly duplicated-K/V MHA (tiny sizes)."""
    B, L, h_q, g, d = 1, 4, 4, 2, 3
    G = h_q // g
    q = _rand((B, L, h_q, d), 41)
    k = _rand((B, L, g, d), 42)
    v = _rand((B, L, g, d), 43)
    scale = 0.7
    for causal in (False, True):
        o, lse = oracle.prefill(q, k, v, causal, scale)
        for h in range(h_q):
            kv = h // G
            for i in range(L):
                js = [j for j in range(L) if (not causal or j <= i)]
                s = [scale * sum(q[0, i, h, t] * k[0, j, kv, t] for t in range(d)) for j in js]
                mx = max(s)
                w = [math.exp(x - mx) for x in s]
                tot = sum(w)
                for t in range(d):
                    ref = sum(w[n] * v[0, js[n], kv, t] for n in range(len(js))) / tot
                    assert abs(o[0, i, h, t] - ref) < 1e-12
                assert abs(lse[0, h, i] - (mx + math.log(tot))) < 1e-12


def test_mha_special_case_identity_map():
    B, L, h, d = 2, 6, 4, 8
    assert list(oracle.head_map(h, h)) == list(range(h))
    q = _rand((B, L, h, d), 51)
    k = _rand((B, L, h, d), 52)
    v = _rand((B, L, h, d), 53)
    o, _ = oracle.prefill(q, k, v, True, 0.4)
    # per-head library attention with no grouping at all
    ref = F.scaled_dot_product_attention(
        torch.from_numpy(q).transpose(1, 2), torch.from_numpy(k).transpose(1, 2),
        torch.from_numpy(v).transpose(1, 2), is_causal=True, scale=0.4)
    np.testing.assert_allclose(o, ref.transpose(1, 2).numpy(), rtol=0, atol=1e-12)


def test_mqa_special_case_expand_form():
    """g = 1: every query head attends to the single K/V head (broadcast form)."""
    B, L, h, d = 2, 5, 6, 8
    assert list(oracle.head_map(h, 1)) == [0] * h
    q = _rand((B, L, h, d), 61)
    k = _rand((B, L, 1, d), 62)
    v = _rand((B, L, 1, d), 63)
    o, _ = oracle.prefill(q, k, v, False, 0.35)
    kb = np.broadcast_to(k, (B, L, h, d))   # expand, no copy
    vb = np.broadcast_to(v, (B, L, h, d))
    s = np.einsum("bihd,bjhd->bhij", q, kb) * 0.35
    p = np.exp(s - s.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    ref = np.einsum("bhij,bjhd->bihd", p, vb)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


def test_head_map_values():
    assert list(oracle.head_map(8, 2)) == [0, 0, 0, 0, 1, 1, 1, 1]
    assert list(oracle.head_map(32, 8)) == [i // 4 for i in range(32)]
    with pytest.raises(ValueError):
        oracle.head_map(8, 3)


def test_permutation_within_group_only():
    check_permutation_within_group()


def test_rows_sum_to_one_and_causal_zeros():
    check_rows_sum_to_one()


def test_causal_row0_returns_v0_exactly():
    check_causal_row0_is_v0()


def test_constant_v_gives_constant_output():
    q = _rand((1, 7, 4, 8), 71)
    k = _rand((1, 7, 2, 8), 72)
    v = np.full((1, 7, 2, 8), 2.5)
    for causal in (False, True):
        o, _ = oracle.prefill(q, k, v, causal, 1.3)
        np.testing.assert_allclose(o, 2.5, rtol=0, atol=1e-12)


def test_zero_q_gives_prefix_mean():
    L = 6
    q = np.zeros((1, L, 4, 8))
    k = _rand((1, L, 2, 8), 81)
    v = _rand((1, L, 2, 8), 82)
    o, lse = oracle.prefill(q, k, v, True, 1.0)
    for i in range(L):
        for h in range(4):
            np.testing.assert_allclose(o[0, i, h], v[0, :i + 1, h // 2].mean(0), rtol=0, atol=1e-12)
            assert abs(lse[0, h, i] - math.log(i + 1)) < 1e-12


def test_decode_equals_row_of_causal_prefill():
    B, L, h_q, g, d = 2, 9, 8, 2, 16
    q = _rand((B, L, h_q, d), 91)
    k = _rand((B, L, g, d), 92)
    v = _rand((B, L, g, d), 93)
    o, lse = oracle.prefill(q, k, v, True, 0.25)
    kc = np.ascontiguousarray(k.transpose(0, 2, 1, 3))  # [B, g, L, d]
    vc = np.ascontiguousarray(v.transpose(0, 2, 1, 3))
    for t in range(L):
        od, lsed = oracle.decode(q[:, t], kc, vc, np.full(B, t + 1), 0.25)
        np.testing.assert_allclose(od, o[:, t], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lsed, lse[:, :, t], rtol=0, atol=1e-12)


def test_prefill_q_offset_equals_rows_of_full_prefill():
    """Bottom rows of a causal prefill, computed with their position offset."""
    B, L, h_q, g, d = 1, 8, 4, 2, 8
    q = _rand((B, L, h_q, d), 95)
    k = _rand((B, L, g, d), 96)
    v = _rand((B, L, g, d), 97)
    o, lse = oracle.prefill(q, k, v, True, 0.5)
    o3, lse3 = oracle.prefill(q[:, 5:], k, v, True, 0.5, q_offset=5)
    np.testing.assert_allclose(o3, o[:, 5:], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse3, lse[:, :, 5:], rtol=0, atol=1e-12)


def test_decode_ignores_rows_past_length_and_empty_rows():
    B, h_q, g, d, S = 3, 4, 2, 8, 10
    q = _rand((B, h_q, d), 101)
    kc = _rand((B, g, S, d), 102)
    vc = _rand((B, g, S, d), 103)
    lens = np.array([4, 10, 0])
    o, lse = oracle.decode(q, kc, vc, lens, 0.3)
    kc2, vc2 = kc.copy(), vc.copy()
    kc2[0, :, 4:] = np.nan
    vc2[0, :, 4:] = np.inf
    o2, lse2 = oracle.decode(q, kc2, vc2, lens, 0.3)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    assert np.all(o[2] == 0.0) and np.all(np.isneginf(lse[2]))


def test_append_then_decode_equals_decode_on_concatenation():
    B, h_q, g, d, S, T = 2, 4, 2, 8, 12, 3
    kc = _rand((B, g, S, d), 111)
    vc = _rand((B, g, S, d), 112)
    lens = np.array([5, 9])
    kn = _rand((B, T, g, d), 113)
    vn = _rand((B, T, g, d), 114)
    kc2, vc2, lens2, status = oracle.append(kc, vc, lens, kn, vn)
    assert status == oracle.APPEND_OK and list(lens2) == [8, 12]
    q = _rand((B, h_q, d), 115)
    o, _ = oracle.decode(q, kc2, vc2, lens2, 0.35)
    for b in range(B):
        kcat = np.concatenate([kc[b, :, :lens[b]], kn[b].transpose(1, 0, 2)], axis=1)
        vcat = np.concatenate([vc[b, :, :lens[b]], vn[b].transpose(1, 0, 2)], axis=1)
        ob, _ = oracle.decode(q[b:b + 1], kcat[None], vcat[None], [lens[b] + T], 0.35)
        np.testing.assert_allclose(o[b], ob[0], rtol=0, atol=1e-12)


def test_bf16_conversions_match_torch():
    x = torch.randn(4096, dtype=torch.float32) * 7
    # include exact ties between two bf16 numbers
    ties = torch.tensor([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(2.0 + 2 ** -7)], dtype=torch.float32)
    x = torch.cat([x, ties])
    b = x.to(torch.bfloat16)
    bits = b.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.f32_to_bf16_bits(x.numpy()), bits)
    assert np.array_equal(oracle.bf16_bits_to_f64(bits), b.to(torch.float64).numpy())


# ---------------------------------------------------------------------------
# Mutation tests: a planted mistake must fail at least one pin
# ---------------------------------------------------------------------------

def _tile_heads(x, group_size, axis):
    # the ``.repeat`` reading: heads tiled, so query head i reads i % g
    reps = [1] * x.ndim
    reps[axis] = group_size
    return np.tile(x, reps)


def _softmax_wrong_axis(scores):
    m = np.max(scores, axis=-1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(scores - m)
    s = np.sum(e, axis=0, keepdims=True)
    return e / s, m, np.sum(e, axis=-1, keepdims=True)


MUTANTS = {
    "modulo_head_map": ("_expand_kv", _tile_heads),
    "causal_off_by_one": ("_visible", lambda i, j, off, window=0: j < i + off),
    "window_off_by_one": ("_visible",
                          lambda i, j, off, window=0: j <= i + off and
                          (window <= 0 or j >= i + off - window)),
    "alibi_wrong_sign": ("_alibi_bias",
                         lambda n_q, n_k, slope, off: slope * np.abs(
                             np.arange(n_q)[:, None] + off - np.arange(n_k)[None, :])),
    "softmax_wrong_axis": ("_softmax_rows", _softmax_wrong_axis),
    "lse_without_max": ("_lse", lambda m, s: np.log(s)),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(gqa_oracle, attr, fn)
    caught = 0
    for chk in _all_checks():
        try:
            chk()
        except (AssertionError, ValueError, IndexError):
            caught += 1
    assert caught >= 1, f"mutant {name} passed every pin"


# ---------------------------------------------------------------------------
# Score-bias variants and chunked prefill over a cache
# ---------------------------------------------------------------------------

def test_window_matches_library_sdpa_with_band_mask():
    check_window_against_sdpa_mask()


def test_window_one_returns_own_v_exactly():
    check_window_one_returns_own_v()


def test_window_at_least_the_length_is_plain_causal():
    q, k, v = _rand((1, 7, 4, 8), 71), _rand((1, 7, 2, 8), 72), _rand((1, 7, 2, 8), 73)
    o_w, l_w = oracle.prefill(q, k, v, True, 0.3, window=7)
    o, l = oracle.prefill(q, k, v, True, 0.3)
    np.testing.assert_array_equal(o_w, o)
    np.testing.assert_array_equal(l_w, l)


def test_window_requires_causal():
    q, k = _rand((1, 3, 2, 4), 74), _rand((1, 3, 1, 4), 75)
    with pytest.raises(ValueError):
        oracle.prefill(q, k, k, False, 0.5, window=2)


def test_alibi_causal_matches_library_sdpa_on_augmented_vectors():
    check_alibi_causal_against_sdpa_augmented()


def test_alibi_zero_slopes_is_plain_attention():
    q, k, v = _rand((2, 6, 4, 8), 81), _rand((2, 6, 2, 8), 82), _rand((2, 6, 2, 8), 83)
    for causal in (True, False):
        o_a, l_a = oracle.prefill(q, k, v, causal, 0.3, alibi_slopes=np.zeros(4))
        o, l = oracle.prefill(q, k, v, causal, 0.3)
        np.testing.assert_allclose(o_a, o, rtol=0, atol=1e-15)
        np.testing.assert_allclose(l_a, l, rtol=0, atol=1e-15)


def test_alibi_noncausal_brute_force_loops():
    B, L, h_q, g, d = 1, 4, 4, 2, 3
    q, k, v = _rand((B, L, h_q, d), 91), _rand((B, L, g, d), 92), _rand((B, L, g, d), 93)
    slopes = [0.5, 0.25, 0.125, 0.0625]
    scale = 0.7
    o, lse = oracle.prefill(q, k, v, False, scale, alibi_slopes=np.array(slopes))
    for h in range(h_q):
        kv = h // (h_q // g)
        for i in range(L):
            w = [math.exp(scale * sum(q[0, i, h, c] * k[0, j, kv, c] for c in range(d))
                          - slopes[h] * abs(i - j)) for j in range(L)]
            tot = sum(w)
            for c in range(d):
                ref = sum(w[j] * v[0, j, kv, c] for j in range(L)) / tot
                assert abs(o[0, i, h, c] - ref) < 1e-12
            assert abs(lse[0, h, i] - math.log(tot)) < 1e-12


def test_prefill_cached_equals_tail_of_full_causal_prefill():
    B, T, h_q, g, d, S_max = 3, 4, 8, 2, 8, 13
    lens = [9, 4, 13]
    rng_seed = 101
    for window, alibi in ((0, None), (3, None), (0, [2.0 ** -(h + 1) for h in range(h_q)]),
                          (5, [0.3] * h_q)):
        kc, vc = _rand((B, g, S_max, d), rng_seed), _rand((B, g, S_max, d), rng_seed + 1)
        q_full = _rand((B, S_max, h_q, d), rng_seed + 2)
        q_new = np.stack([q_full[b, lens[b] - T:lens[b]] for b in range(B)])
        slopes = None if alibi is None else np.array(alibi)
        o, lse = oracle.prefill_cached(q_new, kc, vc, lens, 0.35, window=window,
                                       alibi_slopes=slopes)
        for b in range(B):
            n = lens[b]
            k_full = kc[b:b + 1, :, :n].transpose(0, 2, 1, 3)
            v_full = vc[b:b + 1, :, :n].transpose(0, 2, 1, 3)
            o_f, l_f = oracle.prefill(q_full[b:b + 1, :n], k_full, v_full, True, 0.35,
                                      window=window, alibi_slopes=slopes)
            np.testing.assert_allclose(o[b], o_f[0, n - T:], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse[b], l_f[0, :, n - T:], rtol=0, atol=1e-12)


def test_decode_with_window_and_alibi_is_one_token_chunk():
    B, h_q, g, d, S_max = 3, 8, 4, 8, 12
    kc, vc = _rand((B, g, S_max, d), 111), _rand((B, g, S_max, d), 112)
    q = _rand((B, h_q, d), 113)
    lens = [12, 5, 1]
    slopes = np.array([2.0 ** (-8.0 * (h + 1) / h_q) for h in range(h_q)])
    for window in (0, 1, 4):
        for al in (None, slopes):
            o, lse = oracle.decode(q, kc, vc, lens, 0.4, window=window, alibi_slopes=al)
            o_c, l_c = oracle.prefill_cached(q[:, None], kc, vc, lens, 0.4, window=window,
                                             alibi_slopes=al)
            np.testing.assert_allclose(o, o_c[:, 0], rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse, l_c[:, :, 0], rtol=0, atol=1e-12)


def test_decode_window_equals_decode_over_the_last_rows():
    # ALiBi depends on distance only, so moving the window's rows to the
    # front of a shorter cache leaves the result unchanged
    B, h_q, g, d, S_max, W = 2, 4, 2, 8, 10, 3
    kc, vc = _rand((B, g, S_max, d), 121), _rand((B, g, S_max, d), 122)
    q = _rand((B, h_q, d), 123)
    lens = [10, 7]
    slopes = np.array([0.5, 0.25, 0.125, 0.0625])
    o, _ = oracle.decode(q, kc, vc, lens, 0.5, window=W, alibi_slopes=slopes)
    for b in range(B):
        n = lens[b]
        o_t, _ = oracle.decode(q[b:b + 1], kc[b:b + 1, :, n - W:n], vc[b:b + 1, :, n - W:n],
                               [W], 0.5, alibi_slopes=slopes)
        np.testing.assert_allclose(o[b], o_t[0], rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Paged KV cache
# ---------------------------------------------------------------------------

def _paged_from_contiguous(kc, page_size, perm_seed=None):
    """Split a contiguous [B, g, S, d] cache into pages; optionally shuffle them."""
    B, g, S, d = kc.shape
    nb = S // page_size
    # page b*nb + i holds rows i*page_size .. of sequence b (reshape, no loops)
    pool = kc.reshape(B, g, nb, page_size, d).transpose(0, 2, 1, 3, 4).reshape(B * nb, g,
                                                                                page_size, d)
    table = np.arange(B * nb).reshape(B, nb)
    if perm_seed is not None:
        perm = np.random.default_rng(perm_seed).permutation(B * nb)
        new_pool = np.empty_like(pool)
        new_pool[perm] = pool          # page p moves to slot perm[p]
        pool, table = new_pool, perm[table]
    return pool, table


def test_paged_decode_with_identity_table_equals_contiguous_decode():
    B, h_q, g, d, S, P = 3, 8, 2, 8, 64, 16
    kc, vc, q = _rand((B, g, S, d), 131), _rand((B, g, S, d), 132), _rand((B, h_q, d), 133)
    lens = [64, 17, 1]
    kp, table = _paged_from_contiguous(kc, P)
    vp, _ = _paged_from_contiguous(vc, P)
    o, lse = oracle.decode_paged(q, kp, vp, table, lens, P, 0.3)
    o_c, lse_c = oracle.decode(q, kc, vc, lens, 0.3)
    np.testing.assert_array_equal(o, o_c)
    np.testing.assert_array_equal(lse, lse_c)


def test_paged_decode_is_invariant_to_page_placement():
    B, h_q, g, d, S, P = 2, 4, 4, 8, 48, 16
    kc, vc, q = _rand((B, g, S, d), 141), _rand((B, g, S, d), 142), _rand((B, h_q, d), 143)
    lens = [40, 48]
    slopes = np.array([0.5, 0.25, 0.125, 0.0625])
    kp, table = _paged_from_contiguous(kc, P, perm_seed=7)
    vp, table_v = _paged_from_contiguous(vc, P, perm_seed=7)
    assert np.array_equal(table, table_v)
    for window, al in ((0, None), (20, slopes)):
        o, _ = oracle.decode_paged(q, kp, vp, table, lens, P, 0.3, window=window,
                                   alibi_slopes=al)
        o_c, _ = oracle.decode(q, kc, vc, lens, 0.3, window=window, alibi_slopes=al)
        np.testing.assert_array_equal(o, o_c)


def test_paged_append_matches_contiguous_append():
    B, g, d, S, P, T = 2, 2, 4, 32, 8, 5
    kc, vc = _rand((B, g, S, d), 151), _rand((B, g, S, d), 152)
    kn, vn = _rand((B, T, g, d), 153), _rand((B, T, g, d), 154)
    lens = np.array([30, 6])  # sequence 0 overflows its 32-row capacity
    kp, table = _paged_from_contiguous(kc, P, perm_seed=3)
    vp, _ = _paged_from_contiguous(vc, P, perm_seed=3)
    kp2, vp2, lens_p, st_p = oracle.append_paged(kp, vp, table, lens, kn, vn, P)
    kc2, vc2, lens_c, st_c = oracle.append(kc, vc, lens, kn, vn)
    assert st_p == st_c == oracle.APPEND_CACHE_FULL
    assert list(lens_p) == list(lens_c) == [32, 11]
    np.testing.assert_array_equal(oracle.gather_paged(kp2, table, lens_p, P), kc2 * (
        np.arange(S)[None, None, :, None] < lens_c[:, None, None, None]))
