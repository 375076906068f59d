"""The guard-band helper the GPU tests use, checked on CPU tensors: it must
see a write just past either end of the guarded tensor and nothing else."""

import torch

import guard


def test_guard_detects_writes_past_either_end():
    for dtype in (torch.float32, torch.bfloat16):
        g = guard.empty((3, 5, 7), dtype, "cpu")
        assert torch.isnan(g.tensor.float()).all()  # unwritten outputs read as NaN
        g.tensor.fill_(1.0)
        assert g.bands_intact()
        g.raw[g.pad + g.n] = 0  # first element after the tensor
        assert not g.bands_intact()
        g2 = guard.empty((4,), dtype, "cpu")
        g2.raw[g2.pad - 1] = 0  # last element before it
        assert not g2.bands_intact()


def test_guarded_copy_keeps_the_data_and_alignment():
    t = torch.arange(24, dtype=torch.int32).view(2, 3, 4)
    g = guard.copy_of(t)
    assert torch.equal(g.tensor, t) and g.tensor.is_contiguous()
    assert g.tensor.data_ptr() % 16 == 0
    assert g.bands_intact()
