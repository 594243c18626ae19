"""Seeded synthetic inputs, shared by the oracle tests and the CUDA path.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no norm, no quantization, no dot product).  Each stream
is a numpy PCG64 generator keyed by (workload seed, stream name), so any
consumer can regenerate exactly the same fp32 arrays.

Distributions (the sources measure real Llama-family checkpoints, which are
not available here; these stand in for them):
  * weights      ~ N(0, 0.02)          fp32 [O][K]
  * activations  ~ N(0, 1)             fp32 [N][K], optional outliers: a
                   fraction of the entries of each vector, chosen uniformly
                   without replacement, multiplied by a factor (20)
  * gamma        ~ U(0.5, 1.5)         fp32 [K]
  * raw bytes    ~ U{0..255}            uint8, for large block-format inputs
                   whose fields need no particular distribution
"""
from __future__ import annotations

import zlib

import numpy as np


def _gen(seed: int, stream: str) -> np.random.Generator:
    key = zlib.crc32(stream.encode("utf-8"))
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), key])))


def weights(seed: int, name: str, rows: int, cols: int, sigma: float = 0.02,
            row_begin: int = 0, row_end: int | None = None) -> np.ndarray:
    """fp32 [rows][cols] ~ N(0, sigma).  ``row_begin/row_end`` select a row range
    of the same matrix without drawing the rest (rows are drawn in fixed
    chunks, so any sub-range is reproducible)."""
    if row_end is None:
        row_end = rows
    chunk = 1024
    out = np.empty((row_end - row_begin, cols), dtype=np.float32)
    c0 = row_begin // chunk
    c1 = (row_end + chunk - 1) // chunk
    for c in range(c0, c1):
        g = _gen(seed, f"W:{name}:{c}")
        lo = c * chunk
        hi = min(rows, lo + chunk)
        blk = g.standard_normal((hi - lo, cols), dtype=np.float32)
        blk *= np.float32(sigma)
        a = max(lo, row_begin)
        b = min(hi, row_end)
        if a < b:
            out[a - row_begin:b - row_begin] = blk[a - lo:b - lo]
    return out


def weight_rows(seed: int, name: str, rows: int, cols: int, index: np.ndarray,
                sigma: float = 0.02) -> np.ndarray:
    """fp32 rows ``index`` (sorted) of the matrix ``weights(seed, name, rows, cols)``,
    drawing only the chunks that contain them."""
    index = np.asarray(index, dtype=np.int64)
    out = np.empty((index.shape[0], cols), dtype=np.float32)
    chunk = 1024
    for c in np.unique(index // chunk):
        sel = np.nonzero(index // chunk == c)[0]
        lo = int(c) * chunk
        hi = min(rows, lo + chunk)
        blk = weights(seed, name, rows, cols, sigma=sigma, row_begin=lo, row_end=hi)
        out[sel] = blk[index[sel] - lo]
    return out


def activations(seed: int, name: str, n: int, cols: int, outlier_frac: float = 0.0,
                outlier_mult: float = 20.0) -> np.ndarray:
    """fp32 [n][cols] ~ N(0, 1) with optional per-vector outliers."""
    g = _gen(seed, f"x:{name}")
    x = g.standard_normal((n, cols), dtype=np.float32)
    n_out = int(np.floor(outlier_frac * cols))
    if n_out > 0:
        for i in range(n):
            idx = g.choice(cols, size=n_out, replace=False)
            x[i, idx] *= np.float32(outlier_mult)
    return x


def gamma(seed: int, name: str, cols: int) -> np.ndarray:
    """fp32 [cols] ~ U(0.5, 1.5)."""
    g = _gen(seed, f"gamma:{name}")
    return g.uniform(0.5, 1.5, size=cols).astype(np.float32)


def raw_bytes(seed: int, name: str, count: int) -> np.ndarray:
    """uint8 [count], uniform over 0..255 (stand-in bytes of a block format
    whose every field is then valid or overwritten by the caller)."""
    return _gen(seed, name).integers(0, 256, size=count, dtype=np.uint8)


def sample_indices(seed: int, name: str, total: int, count: int) -> np.ndarray:
    """Sorted distinct indices in [0, total) used to sample outputs for checks."""
    g = _gen(seed, f"sample:{name}")
    count = min(count, total)
    return np.sort(g.choice(total, size=count, replace=False)).astype(np.int64)
