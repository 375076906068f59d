"""Guard bands around device buffers: a check that no kernel writes outside
the tensors it is given.

Each guarded tensor is a view into the middle of a larger allocation whose
leading and trailing bands hold a NaN bit pattern (a payload no kernel
produces). After the library call the bands must still hold that exact
pattern, byte for byte. Output buffers can also be pre-filled with the same
pattern, so an element the kernel should have written but did not stays NaN
and fails the parity comparison.

compute-sanitizer is not available on the GPU machines these tests run on;
the bands stand in for its out-of-bounds write check on the buffers the
library writes (outputs, lse, caches and page pools).
"""

from __future__ import annotations

import math

import torch

BAND_BYTES = 256 << 10  # per side; larger than one prefill output tile (128 rows x 512 B)
CANARY_32 = 0x7FC0DEAD  # fp32 quiet NaN with a payload
CANARY_16 = 0x7FDE      # bf16 quiet NaN with a payload


class Guarded:
    """A tensor inside a canary-filled allocation."""

    def __init__(self, shape, dtype, device, init: torch.Tensor | None = None,
                 band_bytes: int = BAND_BYTES):
        es = torch.empty((), dtype=dtype).element_size()
        if es == 4:
            word, canary = torch.int32, CANARY_32
        elif es == 2:
            word, canary = torch.int16, CANARY_16
        else:
            raise TypeError(f"no canary for {dtype}")
        self.n = math.prod(shape)
        self.pad = band_bytes // es
        self.canary = canary
        raw = torch.full((self.n + 2 * self.pad,), canary, dtype=torch.int64, device=device)
        self.raw = raw.to(word)
        self.tensor = self.raw.view(dtype)[self.pad:self.pad + self.n].view(shape)
        if init is not None:
            self.tensor.copy_(init)

    def bands_intact(self) -> bool:
        if self.raw.is_cuda:
            torch.cuda.synchronize()
        lo = self.raw[:self.pad]
        hi = self.raw[self.pad + self.n:]
        c = torch.tensor(self.canary, dtype=torch.int64).to(self.raw.dtype).item()
        return bool(torch.all(lo == c).item()) and bool(torch.all(hi == c).item())

    def assert_bands(self, what: str):
        assert self.bands_intact(), f"{what}: a kernel wrote outside the buffer (guard band)"


def empty(shape, dtype, device) -> Guarded:
    """An output buffer pre-filled with the canary (unwritten elements stay NaN)."""
    return Guarded(shape, dtype, device)


def copy_of(t: torch.Tensor) -> Guarded:
    """A guarded copy of t (for buffers the library updates in place)."""
    return Guarded(tuple(t.shape), t.dtype, t.device, init=t)
