"""The kernels' failure path on the device, without a fault.

Every wait in the library's kernels is bounded; a wait that runs out makes
the kernel stop and write GQA_ERR_TIMEOUT to the status word. The self-test
entry point runs that wait against a barrier nothing arrives at: the status
must read TIMEOUT, a status that already held an error keeps it (first error
wins), and the device keeps working afterwards.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from grouped_query_attention_10_b300 import binding as gqa
from grouped_query_attention_10_b300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_bounded_wait_runs_out_and_reports_timeout():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gqa.gqa_selftest_bounded_wait(status, limit_us=2000)
    torch.cuda.synchronize()
    assert int(status.item()) == gqa.GQA_ERR_TIMEOUT


def test_first_error_is_kept():
    status = torch.full((1,), gqa.GQA_ERR_CACHE_FULL, dtype=torch.int32, device=DEV)
    gqa.gqa_selftest_bounded_wait(status, limit_us=500)
    torch.cuda.synchronize()
    assert int(status.item()) == gqa.GQA_ERR_CACHE_FULL


def test_device_keeps_working_after_a_timeout():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gqa.gqa_selftest_bounded_wait(status, limit_us=1000)
    torch.cuda.synchronize()
    assert int(status.item()) == gqa.GQA_ERR_TIMEOUT
    B, h_q, g, d, S = 2, 16, 4, 128, 700
    q = inputs.random_bf16((B, h_q, d), 5, device="cpu").to(DEV)
    kc = inputs.random_bf16((B, g, S, d), 6, device="cpu").to(DEV)
    vc = inputs.random_bf16((B, g, S, d), 7, device="cpu").to(DEV)
    lens = torch.tensor([700, 123], dtype=torch.int32, device=DEV)
    fresh = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = gqa.gqa_decode_fwd(q, kc, vc, lens, status=fresh)
    torch.cuda.synchronize()
    assert int(fresh.item()) == 0
    f64 = lambda t: t.detach().cpu().double().numpy()
    o_ref, _ = oracle.decode(f64(q), f64(kc), f64(vc), [700, 123], 1.0 / math.sqrt(d))
    assert np.abs(f64(o) - o_ref).max() <= 1e-2
