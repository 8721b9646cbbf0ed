"""Helpers shared by the GPU tests: moving bf16 bit patterns between numpy
and CUDA tensors, and the parity criterion |y - y_ref| <= 2^-7 |y_ref| + 1e-3
(NaN or Inf fail)."""
import numpy as np
import torch

REL_TOL = 2.0 ** -7
ABS_TOL = 1e-3


def up(bits, dev="cuda"):
    if bits is None:
        return None
    if bits.dtype == np.uint8:
        return torch.from_numpy(np.ascontiguousarray(bits)).to(dev)
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


def down(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def widen(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def mismatches(got_bits, ref_bits):
    g, r = widen(got_bits), widen(ref_bits)
    return ~(np.isfinite(g) & np.isfinite(r) & (np.abs(g - r) <= REL_TOL * np.abs(r) + ABS_TOL))


def assert_parity(got_bits, ref_bits, what=""):
    got_bits = np.asarray(got_bits)
    ref_bits = np.asarray(ref_bits)
    assert got_bits.shape == ref_bits.shape, (got_bits.shape, ref_bits.shape)
    bad = mismatches(got_bits, ref_bits)
    if bad.any():
        idx = np.argwhere(bad)[:8]
        g, r = widen(got_bits), widen(ref_bits)
        detail = ", ".join(f"{tuple(i)}: got {g[tuple(i)]:.6g} want {r[tuple(i)]:.6g}" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; {detail}")


def empty_bf16(*shape):
    return torch.empty(*shape, dtype=torch.bfloat16, device="cuda")


def poison_bf16(*shape):
    # NaN-filled output: an element the kernel forgets to write fails parity.
    return torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
