"""Workload shapes: the decode, small-batch and prefill problems the kernels serve.

Pure data, no arithmetic of the method.  Every shape here is a Llama-style
projection (rows = output features O, columns = input features K) taken from
the model families the sources name when they measure decode speed
(Llama-3.2-1B, an 8B-class Llama, a hidden size of 4096 with a 14336 FFN)
[llama.cpp b10981: OpenVINO backend optimises stateful decode and GPU MoE
inference, section "KV state reorder ... 6.27 -> 9.11 t/s"].

A decode step runs one matrix-vector product per projection
[GGML: Backend abstraction and hardware acceleration, section "CUDA: mmvq,
mmq, cublas -- three matrix paths" (batch-1 decode takes the mmvq route)].
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class Matrix:
    """One quantized projection: ``rows`` outputs over ``cols`` inputs."""

    name: str
    rows: int          # O
    cols: int          # K
    # Which activation feeds it: "norm:<tag>" = fused RMSNorm*gamma -> Q8_0 of
    # activation <tag>; "plain:<tag>" = Q8_0 of activation <tag> with no norm.
    source: str


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    matrices: tuple
    # activation tag -> length K
    activations: dict = field(default_factory=dict)
    n_cols: int = 1                   # N (vectors per call)
    outlier_frac: float = 0.0         # fraction of entries multiplied by outlier_mult
    outlier_mult: float = 20.0
    eps: float = 1e-6


def _mk(name, seed, mats, n_cols=1, outlier_frac=0.0):
    acts = {}
    for m in mats:
        tag = m.source.split(":", 1)[1]
        acts.setdefault(tag, m.cols)
        assert acts[tag] == m.cols, (tag, acts[tag], m.cols)
    return Workload(name=name, seed=seed, matrices=tuple(mats), activations=acts,
                    n_cols=n_cols, outlier_frac=outlier_frac)


# 256 x 256, one vector, fused norm: the parity case the oracle finishes instantly.
TINY = _mk("tiny", 0, [Matrix("w", 256, 256, "norm:x")])

# Llama-3.2-1B-shaped decode step, batch 1 (hidden 2048, GQA k/v 512, FFN 8192).
# The down projection takes a plain-quantized input (no norm in front of it).
LLAMA_1B = _mk("llama-1b-decode", 1, [
    Matrix("q", 2048, 2048, "norm:attn"),
    Matrix("k", 512, 2048, "norm:attn"),
    Matrix("v", 512, 2048, "norm:attn"),
    Matrix("gate", 8192, 2048, "norm:ffn"),
    Matrix("up", 8192, 2048, "norm:ffn"),
    Matrix("down", 2048, 8192, "plain:h"),
])

# 8B-shaped decode step, batch 1: hidden 4096, FFN 14336, GQA k/v 1024, vocab
# head 128256; activations carry 1% outliers x20.  The attention output
# projection o takes a plain-quantized input, as does down.
LLAMA_8B = _mk("llama-8b-decode", 2, [
    Matrix("q", 4096, 4096, "norm:attn"),
    Matrix("k", 1024, 4096, "norm:attn"),
    Matrix("v", 1024, 4096, "norm:attn"),
    Matrix("o", 4096, 4096, "plain:attn_out"),
    Matrix("gate", 14336, 4096, "norm:ffn"),
    Matrix("up", 14336, 4096, "norm:ffn"),
    Matrix("down", 4096, 14336, "plain:h"),
    Matrix("head", 128256, 4096, "norm:final"),
], outlier_frac=0.01)

# Small-batch decode: N in {2, 4, 8} columns through the two FFN shapes.
SMALL_N_SHAPES = ((14336, 4096), (4096, 14336))
SMALL_N_COLS = (2, 4, 8)
SMALL_N_SEED = 3

# Prefill (mmq-style): Q8_0 activations ~N(0,1), plain-quantized, T tokens.
PREFILL_SHAPES = ((14336, 4096, 512), (4096, 4096, 2048))   # (O, K, T)
PREFILL_SEED = 4

ALL = {w.name: w for w in (TINY, LLAMA_1B, LLAMA_8B)}


def q4_0_bytes(rows: int, cols: int) -> int:
    """Bytes of a Q4_0 matrix: 18 bytes per 32 weights."""
    return rows * (cols // 32) * 18


def q8_0_bytes(n: int, cols: int) -> int:
    """Bytes of n Q8_0 vectors: 34 bytes per 32 values."""
    return n * (cols // 32) * 34


def gemv_algorithmic_bytes(rows: int, cols: int, n: int = 1) -> int:
    """Bytes a GEMV call must move at least once: W + xq + y (fp32)."""
    return q4_0_bytes(rows, cols) + q8_0_bytes(n, cols) + 4 * rows * n
