"""GPU parity of the RoPE append (rotary embedding fused into the cache write).

The fused kernel's cache rows, rotated queries and lengths are compared bit
for bit with the oracle's binary32 evaluation of the survey's RoPE code, on
contiguous and paged caches, in place and out of place, with overflow; then a
serving pipeline (prompt, chunk, decode token) that takes its queries and
keys only through the fused append is compared with the fp64 oracle run on
its own rotated tensors.
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

DEV = "cuda"


def rand_bf16(shape, seed):
    return inputs.random_bf16(shape, seed, device="cpu").to(DEV)


def tables(n_pos, d, base=10000.0):
    inv = base ** (-np.arange(0, d, 2, dtype=np.float64) / d)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("h_q,g", [(32, 8), (8, 8), (32, 1)])
@pytest.mark.parametrize("in_place", [True, False])
def test_rope_append_bit_exact(d, h_q, g, in_place):
    B, T, S_max = 4, 37, 300
    lens0 = [0, 100, 290, 263]  # the third overflows (rows 300.. dropped)
    cos, sin = tables(S_max, d)
    kc = rand_bf16((B, g, S_max, d), 1)
    vc = rand_bf16((B, g, S_max, d), 2)
    kn = rand_bf16((B, T, g, d), 3)
    vn = rand_bf16((B, T, g, d), 4)
    q = rand_bf16((B, T, h_q, d), 5)
    q_before = q.clone()
    q_out = q if in_place else torch.full_like(q, 7.0)
    q_out_before = q_out.clone()
    k_ref, v_ref, l_ref, st_ref, q_ref = oracle.append_rope(
        bits(kc), bits(vc), lens0, bits(kn), bits(vn), cos, sin, q=bits(q_before),
        q_out=bits(q_out_before))
    lens = torch.tensor(lens0, dtype=torch.int32, device=DEV)
    gk, gv = guard.copy_of(kc), guard.copy_of(vc)
    kc, vc = gk.tensor, gv.tensor
    if not in_place:
        gq = guard.copy_of(q_out)
        q_out = gq.tensor
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    res = gqa.kv_cache_append_rope(kc, vc, lens, kn, vn, dev(cos), dev(sin), q=q, q_out=q_out,
                                   status=status)
    torch.cuda.synchronize()
    gk.assert_bands("RoPE append K cache")
    gv.assert_bands("RoPE append V cache")
    if not in_place:
        gq.assert_bands("RoPE append rotated queries")
    assert res is q_out
    assert int(status.item()) == st_ref == oracle.APPEND_CACHE_FULL
    assert list(lens.cpu().numpy()) == list(l_ref)
    assert np.array_equal(bits(kc), k_ref), "rotated keys differ"
    assert np.array_equal(bits(vc), v_ref), "values differ"
    assert np.array_equal(bits(q_out), q_ref), "rotated queries differ"
    if not in_place:
        assert torch.equal(q, q_before)


def test_rope_append_keys_only_large():
    """Full-size token batch (B 8 x T 512, h_q 32, g 8, d 128): every row bit-exact."""
    B, T, h_q, g, d, S_max = 8, 512, 32, 8, 128, 2048
    cos, sin = tables(S_max, d, base=500000.0)
    kc = torch.zeros((B, g, S_max, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    kn = rand_bf16((B, T, g, d), 11)
    vn = rand_bf16((B, T, g, d), 12)
    q = rand_bf16((B, T, h_q, d), 13)
    lens0 = [0, 1, 511, 512, 1000, 1536, 1535, 77]
    k_ref, v_ref, l_ref, st_ref, q_ref = oracle.append_rope(
        bits(kc), bits(vc), lens0, bits(kn), bits(vn), cos, sin, q=bits(q))
    lens = torch.tensor(lens0, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gqa.kv_cache_append_rope(kc, vc, lens, kn, vn, dev(cos), dev(sin), q=q, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == st_ref == oracle.APPEND_OK
    assert list(lens.cpu().numpy()) == list(l_ref)
    assert np.array_equal(bits(kc), k_ref)
    assert np.array_equal(bits(vc), v_ref)
    assert np.array_equal(bits(q), q_ref)


@pytest.mark.parametrize("page", [16, 64, 256])
def test_paged_rope_append_bit_exact(page):
    B, T, h_q, g, d, max_blocks = 3, 40, 16, 4, 128, 1024 // page
    cap = page * max_blocks
    num_pages = B * max_blocks + 2
    perm = np.random.default_rng(page).permutation(num_pages)[: B * max_blocks]
    table = perm.reshape(B, max_blocks).astype(np.int32)
    cos, sin = tables(cap, d)
    kp = rand_bf16((num_pages, g, page, d), 21)
    vp = rand_bf16((num_pages, g, page, d), 22)
    kn = rand_bf16((B, T, g, d), 23)
    vn = rand_bf16((B, T, g, d), 24)
    q = rand_bf16((B, T, h_q, d), 25)
    lens0 = [0, page - 1, cap - 10]
    k_ref, v_ref, l_ref, st_ref, q_ref = oracle.append_paged_rope(
        bits(kp), bits(vp), table, lens0, bits(kn), bits(vn), page, cos, sin, q=bits(q))
    lens = torch.tensor(lens0, dtype=torch.int32, device=DEV)
    gk, gv = guard.copy_of(kp), guard.copy_of(vp)
    kp, vp = gk.tensor, gv.tensor
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gqa.kv_cache_append_paged_rope(kp, vp, dev(table), lens, kn, vn, dev(cos), dev(sin), q=q,
                                   status=status)
    torch.cuda.synchronize()
    gk.assert_bands(f"paged RoPE append K pool page={page}")
    gv.assert_bands(f"paged RoPE append V pool page={page}")
    assert int(status.item()) == st_ref == oracle.APPEND_CACHE_FULL
    assert list(lens.cpu().numpy()) == list(l_ref)
    assert np.array_equal(bits(kp), k_ref)
    assert np.array_equal(bits(vp), v_ref)
    assert np.array_equal(bits(q), q_ref)


def test_rope_pipeline_prompt_chunk_decode():
    """Prompt, chunk and decode token all go through the fused RoPE append
    (queries rotated in place); attention is then compared with the fp64
    oracle on the oracle's own rotated queries and cache."""
    B, h_q, g, d, S_max, P, T = 2, 32, 8, 128, 512, 200, 48
    cos, sin = tables(S_max, d)
    kc = torch.zeros((B, g, S_max, d), dtype=torch.bfloat16, device=DEV)
    vc = torch.zeros_like(kc)
    lens = torch.zeros((B,), dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    k_all = rand_bf16((B, P + T + 1, g, d), 31)
    v_all = rand_bf16((B, P + T + 1, g, d), 32)
    q_all = rand_bf16((B, P + T + 1, h_q, d), 33)
    # the oracle's side, token groups in the same order
    kr, vr, lr = bits(kc), bits(vc), [0] * B
    q_rot = []
    for a, b in ((0, P), (P, P + T), (P + T, P + T + 1)):
        kr, vr, lr, _, qr = oracle.append_rope(kr, vr, lr, bits(k_all[:, a:b].contiguous()),
                                               bits(v_all[:, a:b].contiguous()), cos, sin,
                                               q=bits(q_all[:, a:b].contiguous()))
        q_rot.append(qr)
    # the library's side
    cos_d, sin_d = dev(cos), dev(sin)
    outs = []
    for i, (a, b) in enumerate(((0, P), (P, P + T), (P + T, P + T + 1))):
        qg = q_all[:, a:b].contiguous()
        gqa.kv_cache_append_rope(kc, vc, lens, k_all[:, a:b].contiguous(),
                                 v_all[:, a:b].contiguous(), cos_d, sin_d, q=qg, status=status)
        assert np.array_equal(bits(qg), q_rot[i])
        if i == 1:
            outs.append(gqa.gqa_prefill_kvcache_fwd(qg, kc, vc, lens))
        elif i == 2:
            outs.append(gqa.gqa_decode_fwd(qg[:, 0].contiguous(), kc, vc, lens))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(bits(kc), kr) and np.array_equal(bits(vc), vr)
    scale = 1.0 / math.sqrt(d)
    kv = oracle.bf16_bits_to_f64(kr)
    vv = oracle.bf16_bits_to_f64(vr)
    o_chunk, _ = oracle.prefill_cached(oracle.bf16_bits_to_f64(q_rot[1]), kv, vv, [P + T] * B,
                                       scale)
    o_dec, _ = oracle.decode(oracle.bf16_bits_to_f64(q_rot[2][:, 0]), kv, vv, [P + T + 1] * B,
                             scale)
    for got, ref, what in ((outs[0], o_chunk, "chunk"), (outs[1], o_dec, "decode")):
        err = np.abs(f64(got) - ref)
        assert err.max() <= 1e-2 and err.mean() <= 1e-3, f"{what}: {err.max():.3e}"
