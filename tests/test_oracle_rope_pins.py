"""Pins of the oracle's rotary embedding (RoPE) and of the RoPE append.

The rotation is tied to hand-derived values (tests/golden/rope_closed_form.json),
to properties of a rotation (norm kept, scores depending only on the distance
between positions, position 0 of a true table being a pure reordering), to the
error bound of binary32 arithmetic for the rounded form, and the append to the
plain append, the paged layout and one-token-at-a-time appends. Planted
mistakes (pair layout, sign, position offset) must each fail a pin.
"""

import json
import os

import numpy as np
import pytest

import oracle
from oracle import gqa_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rope_closed_form.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _bits(x):
    return oracle.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _vals(bits):
    return oracle.bf16_bits_to_f64(np.asarray(bits).view(np.uint16))


def _tables(n_pos, d, base=10000.0):
    """True rotation tables: angle p * base^(-2i/d) for pair i at position p."""
    inv = base ** (-np.arange(0, d, 2, dtype=np.float64) / d)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang), np.sin(ang)


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


# --------------------------------------------------------------- the checks

def check_golden_rotation():
    c = _golden()["rotate"]
    x = np.array(c["x"], dtype=np.float64)
    for p, want in enumerate(c["out_by_position"]):
        assert np.array_equal(oracle.rope(x, c["cos"], c["sin"], p), np.array(want, float))
        assert np.array_equal(oracle.rope_f32(x, c["cos"], c["sin"], p).astype(np.float64),
                              np.array(want, float))


def check_golden_append():
    c = _golden()["append"]
    B, g, S, d = c["B"], c["g"], c["S_max"], c["d"]
    gr = _golden()["rotate"]
    kc = _bits(np.full((B, g, S, d), c["cache_fill"]))
    vc = kc.copy()
    kc2, vc2, lens2, status, q2 = oracle.append_rope(
        kc, vc, np.array(c["seq_lens"]), _bits(c["k_new"]), _bits(c["v_new"]),
        gr["cos"], gr["sin"], q=_bits(c["q"]), q_out=_bits(c["q_out_before"]))
    assert np.array_equal(_vals(kc2), np.array(c["k_cache_after"], float))
    assert np.array_equal(_vals(vc2), np.array(c["v_cache_after"], float))
    assert np.array_equal(_vals(q2), np.array(c["q_out_after"], float))
    assert list(lens2) == c["seq_lens_after"]
    assert status == c["status"] == oracle.APPEND_CACHE_FULL


def check_norm_kept():
    cos, sin = _tables(64, 16)
    x = _rand((64, 16), 1)
    y = oracle.rope(x, cos, sin, np.arange(64))
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def check_scores_depend_on_distance_only():
    d = 32
    cos, sin = _tables(300, d)
    q = _rand((d,), 2)
    k = _rand((d,), 3)
    for m, n in [(5, 2), (40, 40), (7, 100)]:
        s0 = oracle.rope(q, cos, sin, m) @ oracle.rope(k, cos, sin, n)
        for shift in (1, 17, 150):
            s1 = oracle.rope(q, cos, sin, m + shift) @ oracle.rope(k, cos, sin, n + shift)
            assert abs(s1 - s0) <= 1e-11 * (1 + abs(s0))


def check_position_zero_is_reordering():
    cos, sin = _tables(4, 8)
    x = _rand((8,), 4)
    assert np.array_equal(oracle.rope(x, cos, sin, 0), np.concatenate([x[0::2], x[1::2]]))


def check_f32_within_binary32_bound():
    d = 64
    cos, sin = _tables(512, d)
    x = _vals(_bits(_rand((512, d), 5) * 3.0))
    pos = np.arange(512)
    exact = oracle.rope(x, cos, sin, pos)
    got = oracle.rope_f32(x, cos, sin, pos).astype(np.float64)
    # tables rounded to binary32 (one half-ulp each), two rounded products and
    # one rounded sum or difference: |err| <= 4 * 2^-24 * (|e||c| + |o||s|) + 2^-24 |out|
    c32 = cos.astype(np.float32).astype(np.float64)[pos]
    s32 = sin.astype(np.float32).astype(np.float64)[pos]
    e, o = np.abs(x[:, 0::2]), np.abs(x[:, 1::2])
    mag = np.concatenate([e * np.abs(c32) + o * np.abs(s32), e * np.abs(s32) + o * np.abs(c32)], -1)
    assert np.all(np.abs(got - exact) <= 4 * 2.0 ** -24 * mag + 2.0 ** -24 * np.abs(exact))


def check_append_rope_is_append_of_rotated_keys():
    B, T, g, h_q, S, d = 3, 5, 2, 4, 12, 8
    cos, sin = _tables(S, d)
    lens = np.array([0, 4, 10])
    kn, vn, q = (_bits(_rand((B, T, n, d), s)) for s, n in ((6, g), (7, g), (8, h_q)))
    kc = _bits(_rand((B, g, S, d), 9))
    vc = _bits(_rand((B, g, S, d), 10))
    kc2, vc2, lens2, st, q2 = oracle.append_rope(kc, vc, lens, kn, vn, cos, sin, q=q)
    # the plain append of the same V rows
    _, vref, lref, stref = oracle.append(vc, vc, lens, vn, vn)
    assert np.array_equal(vc2, vref) and list(lens2) == list(lref) and st == stref
    for b in range(B):
        for t in range(T):
            pos = lens[b] + t
            if pos >= S:
                assert np.array_equal(q2[b, t], q[b, t])
                continue
            want_k = _bits(oracle.rope_f32(_vals(kn[b, t]), cos, sin, pos))
            assert np.array_equal(kc2[b, :, pos], want_k)
            want_q = _bits(oracle.rope_f32(_vals(q[b, t]), cos, sin, pos))
            assert np.array_equal(q2[b, t], want_q)


def check_one_at_a_time_equals_all_at_once():
    B, T, g, S, d = 2, 6, 2, 16, 8
    cos, sin = _tables(S, d)
    lens = np.array([3, 9])
    kn, vn = _bits(_rand((B, T, g, d), 11)), _bits(_rand((B, T, g, d), 12))
    kc = _bits(np.zeros((B, g, S, d)))
    all_k, all_v, all_l, _, _ = oracle.append_rope(kc, kc, lens, kn, vn, cos, sin)
    k1, v1, l1 = kc, kc, lens
    for t in range(T):
        k1, v1, l1, _, _ = oracle.append_rope(k1, v1, l1, kn[:, t:t + 1], vn[:, t:t + 1], cos,
                                              sin)
    assert np.array_equal(all_k, k1) and np.array_equal(all_v, v1)
    assert list(all_l) == list(l1)


def check_paged_matches_contiguous():
    B, T, g, h_q, d, page, nb = 2, 7, 2, 4, 8, 4, 4
    S = page * nb
    cos, sin = _tables(S, d)
    lens = np.array([2, 13])
    kn, vn, q = (_bits(_rand((B, T, n, d), s)) for s, n in ((13, g), (14, g), (15, h_q)))
    table = np.array([[5, 0, 7, 2], [1, 6, 3, 4]])
    pool = _bits(np.zeros((8, g, page, d)))
    kp, vp, lp, stp, qp = oracle.append_paged_rope(pool, pool, table, lens, kn, vn, page, cos,
                                                   sin, q=q)
    kc, vc, lc, stc, qc = oracle.append_rope(_bits(np.zeros((B, g, S, d))),
                                             _bits(np.zeros((B, g, S, d))), lens, kn, vn, cos,
                                             sin, q=q)
    assert np.array_equal(oracle.gather_paged(kp, table, lp, page), kc)
    assert np.array_equal(oracle.gather_paged(vp, table, lp, page), vc)
    assert list(lp) == list(lc) and stp == stc and np.array_equal(qp, qc)


def check_decode_with_rope_depends_on_distances_only():
    # every cached key rotated at its row, the query at the last row: the
    # decode output is the same when all positions move by the same amount
    B, h_q, g, n, d = 1, 4, 2, 20, 16
    cos, sin = _tables(200, d)
    q = _rand((B, h_q, d), 16)
    k = _rand((B, g, n, d), 17)
    v = _rand((B, g, n, d), 18)
    outs = []
    for shift in (0, 37, 150):
        kr = oracle.rope(k, cos, sin, np.arange(n) + shift)
        qr = oracle.rope(q[:, :, None, :], cos, sin, np.array([n - 1 + shift]))[:, :, 0]
        outs.append(oracle.decode(qr, kr, v, [n], 0.25)[0])
    assert np.allclose(outs[0], outs[1], atol=1e-12) and np.allclose(outs[0], outs[2], atol=1e-12)


CHECKS = [check_golden_rotation, check_golden_append, check_norm_kept,
          check_scores_depend_on_distance_only, check_position_zero_is_reordering,
          check_f32_within_binary32_bound, check_append_rope_is_append_of_rotated_keys,
          check_one_at_a_time_equals_all_at_once, check_paged_matches_contiguous,
          check_decode_with_rope_depends_on_distances_only]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_rope_pin(check):
    check()


# ------------------------------------------------ planted mistakes are caught

def _interleaved(x, cos, sin, positions):
    # output pairs kept interleaved instead of split into halves
    x = np.asarray(x, dtype=np.float64)
    c = np.asarray(cos, float)[np.asarray(positions)]
    s = np.asarray(sin, float)[np.asarray(positions)]
    out = np.empty_like(x)
    out[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
    out[..., 1::2] = x[..., 0::2] * s + x[..., 1::2] * c
    return out



def _halves_pairing(x, cos, sin, positions):
    # pairs (i, i + d/2) instead of (2i, 2i + 1)
    x = np.asarray(x, dtype=np.float64)
    h = x.shape[-1] // 2
    c = np.asarray(cos, float)[np.asarray(positions)]
    s = np.asarray(sin, float)[np.asarray(positions)]
    a, b = x[..., :h], x[..., h:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


_ORIG_NEW_ROWS = gqa_oracle._rope_new_rows


def _position_plus_one(x_bits, cos, sin, seq_lens, capacity):
    return _ORIG_NEW_ROWS(x_bits, cos, sin, np.asarray(seq_lens) + 1, capacity)


def _f32_mutant(fn64):
    return lambda x, cos, sin, positions: fn64(x, cos, sin, positions).astype(np.float32)


MUTANTS = {
    "interleaved_output": [("rope", _interleaved), ("rope_f32", _f32_mutant(_interleaved))],
    "halves_pairing": [("rope", _halves_pairing), ("rope_f32", _f32_mutant(_halves_pairing))],
    "negative_angle": [("rope", "neg"), ("rope_f32", "neg32")],
    "position_plus_one": [("_rope_new_rows", _position_plus_one)],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_rope_mistake_is_caught(name, monkeypatch):
    orig = gqa_oracle.rope
    for attr, fn in MUTANTS[name]:
        if fn == "neg":
            fn = lambda x, c, s, p: orig(x, c, -np.asarray(s, float), p)  # noqa: E731
        elif fn == "neg32":
            fn = _f32_mutant(lambda x, c, s, p: orig(x, c, -np.asarray(s, float), p))
        monkeypatch.setattr(gqa_oracle, attr, fn)
        monkeypatch.setattr(oracle, attr, fn, raising=False)
    caught = 0
    for chk in CHECKS:
        try:
            chk()
        except (AssertionError, ValueError, IndexError):
            caught += 1
    assert caught >= 1, f"mutant {name} passed every pin"
