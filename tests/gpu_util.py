"""Helpers for the GPU parity tests: host <-> device transfers and the
tolerance check the attention outputs must meet against the fp64 oracle."""

from __future__ import annotations

import numpy as np
import torch

import workloads as W

# Tolerances for bf16 attention outputs against the fp64 oracle.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def dev():
    return torch.device("cuda:0")


def to_dev(a: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bits (numpy) -> bf16 CUDA tensor."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev()).view(torch.bfloat16)


def to_host(t: torch.Tensor) -> np.ndarray:
    """bf16 CUDA tensor -> uint16 bf16 bits (numpy)."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def i32(a) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev())


def check_close(got_bits: np.ndarray, ref: np.ndarray, what: str, rows=None):
    """bf16 output vs fp64 reference: max-abs <= 2e-2 and mean-abs <= 2e-3."""
    got = W.bf16_bits_to_f32(got_bits).astype(np.float64)
    if rows is not None:
        got, ref = got[rows], ref[rows]
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max-abs {mx:.3g} mean-abs {mean:.3g}"
    return mx, mean


def assert_equal_chunks(a: np.ndarray, b: np.ndarray, what: str, chunk: int = 1 << 26) -> None:
    fa, fb = a.reshape(-1), b.reshape(-1)
    assert fa.size == fb.size
    for lo in range(0, fa.size, chunk):
        if not np.array_equal(fa[lo:lo + chunk], fb[lo:lo + chunk]):
            bad = np.nonzero(fa[lo:lo + chunk] != fb[lo:lo + chunk])[0]
            raise AssertionError(f"{what}: {bad.size} elements differ, first at {lo + int(bad[0])}")
