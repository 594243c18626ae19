"""Shared helpers for the GPU parity tests (inputs, device buffers, checks).

Inputs come from the seeded generators; expected values come only from the
CPU oracle.  The comparison rules:
  * Q8_0 activations and Q4_0 weights: bytes identical (codes and fp16 scales);
  * per-block integer sums: identical;
  * fp32 outputs: |y - y_ref| <= 1e-5 * S elementwise, S = sum_b |d_w d_x isum_b|.
"""
from __future__ import annotations

import numpy as np

TOL = 1e-5


def torch_cuda():
    import torch
    if not torch.cuda.is_available():
        import pytest
        pytest.skip("no CUDA device")
    return torch


def to_dev(a: np.ndarray):
    torch = torch_cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def empty_u8(nbytes: int):
    torch = torch_cuda()
    return torch.empty(nbytes, dtype=torch.uint8, device="cuda")


def to_host(t) -> np.ndarray:
    return t.cpu().numpy()


def assert_within_tol(y_gpu: np.ndarray, y64: np.ndarray, S: np.ndarray, what: str = "y") -> float:
    """Elementwise tolerance; returns the worst |err| / S ratio."""
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    assert y_gpu.shape == y64.shape, (y_gpu.shape, y64.shape)
    assert np.all(np.isfinite(y_gpu)), f"{what}: non-finite output"
    err = np.abs(y_gpu - y64)
    bound = TOL * S
    bad = err > bound
    if np.any(bad):
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} outputs out of tolerance; worst at {i}: "
                             f"gpu={y_gpu[i]!r} ref={y64[i]!r} S={S[i]!r}")
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(S > 0, err / S, 0.0)
    return float(r.max()) if r.size else 0.0
