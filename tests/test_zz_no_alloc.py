"""The allocation-free decode entry point, gqa_decode_fwd_noalloc.

It serves callers that cannot hand the library a workspace -- plugin hosts
whose memory planner owns every allocation, serving loops that must not call
cudaMalloc once running -- from a scratch array built into the library. These
tests call it through the C interface and check that its results match
gqa_decode_fwd (which takes a caller-allocated workspace) on two calls in a
row, the second reusing the scratch left behind by the first, and that they
match the fp64 oracle's decode.

This file is named so that pytest collects it last.
"""

import ctypes

import pytest
import torch

import numpy as np
import oracle
from grouped_query_attention_10_b300 import binding
from grouped_query_attention_10_b300 import inputs

MAX_ABS = 1e-2
MEAN_ABS = 1e-3
FAKE = 1 << 20  # 16-byte-aligned non-null address; never dereferenced


@pytest.fixture(scope="module")
def lib():
    return binding.load_library()


def _noalloc(lib, q, kc, vc, lens, o, lse, B, h_q, g, d, S_max, scale, status=None):
    return lib.gqa_decode_fwd_noalloc(q, kc, vc, lens, o, 0, lse, B, h_q, g, d, S_max, scale,
                                      status, None)


def test_noalloc_scratch_size_and_host_checks(lib):
    """Checks that run before any CUDA call (no device needed)."""
    cap = lib.gqa_decode_noalloc_scratch_bytes()
    assert cap == 32 << 20
    # the ragged decode workload fits: [64, 8, 8192, 128] cache, 32 query heads
    assert 0 < lib.gqa_decode_workspace_bytes(64, 32, 8, 128, 8192) <= cap
    f = FAKE
    assert _noalloc(lib, None, f, f, f, f, None, 4, 32, 8, 128, 1024, 0.1) == binding.GQA_ERR_NULL
    assert _noalloc(lib, f, f, f, f, None, None, 4, 32, 8, 128, 1024, 0.1) == binding.GQA_ERR_NULL
    assert _noalloc(lib, f, f, f, f, f, None, 4, 32, 3, 128, 1024, 0.1) == binding.GQA_ERR_SHAPE
    # sizes needing more scratch than the built-in array are refused
    assert lib.gqa_decode_workspace_bytes(64, 64, 8, 128, 1 << 17) > cap
    assert (_noalloc(lib, f, f, f, f, f, None, 64, 64, 8, 128, 1 << 17, 0.1)
            == binding.GQA_ERR_SCRATCH_LIMIT)
    assert binding.status_string(binding.GQA_ERR_SCRATCH_LIMIT).startswith(
        "GQA_ERR_SCRATCH_LIMIT")


def _close(got, ref, what):
    # an empty sequence has lse = -inf on both paths; everything else is finite
    inf_ref = torch.isneginf(ref)
    assert torch.equal(torch.isneginf(got), inf_ref), f"{what}: -inf entries differ"
    got, ref = got[~inf_ref], ref[~inf_ref]
    assert torch.all(torch.isfinite(got)), what
    err = (got.double() - ref.double()).abs()
    assert err.max().item() <= MAX_ABS, f"{what}: max abs err {err.max().item():.3e}"
    assert err.mean().item() <= MEAN_ABS, f"{what}: mean abs err {err.mean().item():.3e}"


def _case(lib, B, h_q, g, d, S_max, seed, lens_override=None):
    dev = torch.device("cuda", 0)
    w = inputs.DecodeWorkload("noalloc_case", B=B, h_q=h_q, g=g, d=d, S_max=S_max,
                              len_lo=1, len_hi=S_max, seed=seed)
    q, kc, vc, lens = (t.to(dev) for t in inputs.decode_inputs(w))
    if lens_override is not None:
        lens[:len(lens_override)] = torch.tensor(lens_override, dtype=torch.int32)
    scale = 1.0 / d ** 0.5
    # reference: the workspace-taking entry point
    o_ref = torch.empty((B, h_q, d), dtype=torch.float32, device=dev)
    lse_ref = torch.empty((B, h_q), dtype=torch.float32, device=dev)
    binding.gqa_decode_fwd(q, kc, vc, lens, scale=scale, out=o_ref, lse=lse_ref)
    # the allocation-free entry point, through the C interface
    o = torch.full((B, h_q, d), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((B, h_q), float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    rc = _noalloc(lib, q.data_ptr(), kc.data_ptr(), vc.data_ptr(), lens.data_ptr(), o.data_ptr(),
                  lse.data_ptr(), B, h_q, g, d, S_max, ctypes.c_float(scale), status.data_ptr())
    torch.cuda.synchronize()
    assert rc == binding.GQA_OK, binding.status_string(rc)
    assert int(status.item()) == 0
    _close(o, o_ref, f"noalloc O, B={B} g={g} d={d} S_max={S_max}")
    _close(lse, lse_ref, f"noalloc lse, B={B} g={g} d={d} S_max={S_max}")


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_twice(lib):
    # first call: ragged lengths incl. an empty sequence and a full one
    _case(lib, B=8, h_q=32, g=8, d=128, S_max=2048, seed=501, lens_override=[0, 1, 2048, 777])
    # second call in a row: other sizes, reusing the scratch the first call left
    _case(lib, B=3, h_q=16, g=2, d=64, S_max=3000, seed=502, lens_override=[3000, 65])


@pytest.mark.gpu
def test_noalloc_matches_the_oracle(lib):
    dev = torch.device("cuda", 0)
    B, h_q, g, d, S_max = 4, 32, 8, 128, 1000
    w = inputs.DecodeWorkload("noalloc_oracle", B=B, h_q=h_q, g=g, d=d, S_max=S_max,
                              len_lo=1, len_hi=S_max, seed=503)
    q, kc, vc, lens = (t.to(dev) for t in inputs.decode_inputs(w))
    lens_l = [1000, 1, 517, 64]
    lens[:] = torch.tensor(lens_l, dtype=torch.int32)
    scale = 1.0 / d ** 0.5
    o = torch.full((B, h_q, d), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((B, h_q), float("nan"), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    torch.cuda.synchronize()
    rc = _noalloc(lib, q.data_ptr(), kc.data_ptr(), vc.data_ptr(), lens.data_ptr(), o.data_ptr(),
                  lse.data_ptr(), B, h_q, g, d, S_max, ctypes.c_float(scale), status.data_ptr())
    torch.cuda.synchronize()
    assert rc == binding.GQA_OK, binding.status_string(rc)
    assert int(status.item()) == 0
    f64 = lambda t: t.detach().to(torch.float64).cpu().numpy()
    o_ref, lse_ref = oracle.decode(f64(q), f64(kc), f64(vc), lens_l, scale)
    for got, ref, what in ((f64(o), o_ref, "O"), (f64(lse), lse_ref, "lse")):
        err = np.abs(got - ref)
        assert err.max() <= MAX_ABS, f"noalloc {what} vs oracle: max abs err {err.max():.3e}"
        assert err.mean() <= MEAN_ABS, f"noalloc {what} vs oracle: mean abs err {err.mean():.3e}"
