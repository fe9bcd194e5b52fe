"""Shared helpers of the GPU parity tests: tolerance, transfers, guard bands.

Tolerance: |gpu - ref| <= 2e-4 (1 + |ref|) element-wise on y and on the final
states (the parity bound of the mixer core).  A bf16 output is additionally
allowed one bf16 unit in the last place, 2^-8 |ref|, for its single rounding.
"""
import numpy as np
import torch

TOL = 2e-4
BF16_ULP = 2.0 ** -8


def bound(ref, bf16_out=False):
    ref = np.abs(ref)
    b = TOL * (1.0 + ref)
    if bf16_out:
        b = b + BF16_ULP * ref
    return b


def assert_within(got, ref, what, bf16_out=False):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    err = np.abs(got - ref)
    b = bound(ref, bf16_out)
    bad = ~(err <= b)  # NaN counts as bad
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside 2e-4(1+|ref|); "
            f"first at {i}: got {got[i]!r} ref {ref[i]!r}; max err/bound {np.nanmax(err / b):.3g}")
    return float(np.max(err / b)) if err.size else 0.0


def torch_dtype(name):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def to_dev(a, dtype="f32"):
    """Host f32 array (already holding bf16 values when dtype == 'bf16') -> cuda tensor."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()
    return t.to(torch_dtype(dtype)) if dtype != "f32" else t


def to_host(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def strided_copy(a, dtype, ld, offset=0):
    """A [B, T, C] device view with row stride `ld` (elements) into a wider buffer."""
    Bsz, T, C = a.shape
    buf = torch.full((Bsz, T, ld), float("nan"), device="cuda", dtype=torch_dtype(dtype))
    view = buf[:, :, offset:offset + C]
    view.copy_(to_dev(a, dtype))
    return view


class Guarded:
    """A flat device buffer with sentinel guard bands around a [*shape] view."""

    PAD = 4096

    def __init__(self, shape, dtype="f32", fill=7.25):
        n = int(np.prod(shape))
        self.sentinel = fill
        self.buf = torch.full((n + 2 * self.PAD,), fill, device="cuda", dtype=torch_dtype(dtype))
        self.view = self.buf[self.PAD:self.PAD + n].view(*shape)

    def check(self):
        lo = self.buf[: self.PAD]
        hi = self.buf[-self.PAD:]
        assert bool((lo == self.sentinel).all()) and bool((hi == self.sentinel).all()), \
            "write outside the output buffer"
