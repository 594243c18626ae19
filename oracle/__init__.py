"""CPU oracle for the quantized decode GEMV path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and it
shares no code with it.

The arithmetic lives in ``oracle.c`` (plain scalar C, -O2 -ffp-contract=off);
this module compiles it with gcc into ``oracle/_lib/liboracle.so`` and wraps it
with numpy-array helpers.  Every routine cites the passage it follows in
``oracle.c``.  The fp64 tolerance scale ``S`` and the exact block sums make the
comparison rules of the parity tests explicit:

  * quantized activations (q bytes and fp16 scale bits): bit-exact;
  * per-block integer sums: bit-exact;
  * fp32 outputs: |y_gpu - y_ref| <= 1e-5 * S elementwise, S = sum_b |d_w d_x isum_b|.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

QK = 32
Q4_BLOCK = 18
Q8_BLOCK = 34
Q4K_BLOCK = 144          # one Q4_K super-block: 256 weights
Q5K_BLOCK = 176          # one Q5_K super-block: 256 weights
# bytes per 32 weights of each weight type
_BYTES_PER_32 = {"q4_0": Q4_BLOCK, "q8_0": Q8_BLOCK, "q4_k": Q4K_BLOCK // 8, "q5_k": Q5K_BLOCK // 8}


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (host arch, no SIMD flags)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            c_i64, c_f, c_p = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
            L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_f16_to_f32.restype = c_f
            L.orc_f32_to_f16.argtypes = [c_f]
            L.orc_f32_to_f16.restype = ctypes.c_uint16
            L.orc_quantize_q4_0.argtypes = [c_p, c_i64, c_i64, c_p]
            L.orc_quantize_q4_0.restype = None
            L.orc_rms_scale.argtypes = [c_p, c_i64, c_f]
            L.orc_rms_scale.restype = c_f
            L.orc_quantize_q8_0.argtypes = [c_p, c_i64, c_p, c_f, c_i64, c_i64, c_p]
            L.orc_quantize_q8_0.restype = None
            L.orc_quantize_q8_0_add.argtypes = [c_p, c_i64, c_p, c_p, c_i64, c_f, c_i64, c_i64, c_p]
            L.orc_quantize_q8_0_add.restype = None
            L.orc_q4_0_seg_row_bytes.argtypes = [c_i64]
            L.orc_q4_0_seg_row_bytes.restype = c_i64
            L.orc_repack_q4_0_seg.argtypes = [c_p, c_i64, c_i64, c_p]
            L.orc_repack_q4_0_seg.restype = None
            L.orc_block_sums_q8w.argtypes = [c_p, c_p, c_i64, c_i64, c_i64, c_p]
            L.orc_block_sums_q8w.restype = None
            L.orc_matvec_q8w.argtypes = [c_p, c_p, c_i64, c_i64, c_i64, c_p, c_i64, c_p, c_p, c_p]
            L.orc_matvec_q8w.restype = None
            L.orc_block_sums.argtypes = [c_p, c_p, c_i64, c_i64, c_i64, c_p]
            L.orc_block_sums.restype = None
            L.orc_matvec.argtypes = [c_p, c_p, c_i64, c_i64, c_i64, c_p, c_i64, c_p, c_p, c_p]
            L.orc_matvec.restype = None
            L.orc_quantize_q4_k.argtypes = [c_p, c_i64, c_i64, c_p]
            L.orc_quantize_q4_k.restype = None
            L.orc_dequantize_q4_k.argtypes = [c_p, c_i64, c_i64, c_p]
            L.orc_dequantize_q4_k.restype = None
            L.orc_block_sums_q4k.argtypes = [c_p, c_p, c_i64, c_i64, c_i64, c_p]
            L.orc_block_sums_q4k.restype = None
            L.orc_matvec_q4k.argtypes = [c_p, c_p, c_i64, c_i64, c_i64, c_p, c_i64, c_p, c_p, c_p]
            L.orc_matvec_q4k.restype = None
            L.orc_quantize_q5_k.argtypes = [c_p, c_i64, c_i64, c_p]
            L.orc_quantize_q5_k.restype = None
            L.orc_dequantize_q5_k.argtypes = [c_p, c_i64, c_i64, c_p]
            L.orc_dequantize_q5_k.restype = None
            L.orc_block_sums_q5k.argtypes = [c_p, c_p, c_i64, c_i64, c_i64, c_p]
            L.orc_block_sums_q5k.restype = None
            L.orc_matvec_q5k.argtypes = [c_p, c_p, c_i64, c_i64, c_i64, c_p, c_i64, c_p, c_p, c_p]
            L.orc_matvec_q5k.restype = None
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def f16_to_f32(h: int) -> float:
    return float(lib().orc_f16_to_f32(int(h) & 0xFFFF))


def f32_to_f16(f: float) -> int:
    return int(lib().orc_f32_to_f16(float(np.float32(f))))


def quantize_q4_0(w: np.ndarray) -> np.ndarray:
    """fp32 [O][K] -> uint8 [O][K/32*18] (Q4_0 blocks, row-major)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    O, K = w.shape
    assert K % QK == 0
    out = np.empty((O, K // QK * Q4_BLOCK), dtype=np.uint8)
    lib().orc_quantize_q4_0(_ptr(w), O, K, _ptr(out))
    return out


def quantize_q4_k(w: np.ndarray) -> np.ndarray:
    """fp32 [O][K] -> uint8 [O][K/256*144] (Q4_K super-blocks, row-major; see oracle.c)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    O, K = w.shape
    assert K % 256 == 0
    out = np.empty((O, K // 256 * Q4K_BLOCK), dtype=np.uint8)
    lib().orc_quantize_q4_k(_ptr(w), O, K, _ptr(out))
    return out


def dequantize_q4_k(Wq: np.ndarray, K: int) -> np.ndarray:
    """uint8 [O][K/256*144] -> fp64 [O][K], every value d*sc*q - dmin*m exact."""
    Wq = np.ascontiguousarray(np.atleast_2d(Wq), dtype=np.uint8)
    assert K % 256 == 0 and Wq.shape[1] == K // 256 * Q4K_BLOCK
    out = np.empty((Wq.shape[0], K), dtype=np.float64)
    lib().orc_dequantize_q4_k(_ptr(Wq), Wq.shape[0], K, _ptr(out))
    return out


def quantize_q5_k(w: np.ndarray) -> np.ndarray:
    """fp32 [O][K] -> uint8 [O][K/256*176] (Q5_K super-blocks, row-major; see oracle.c)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    O, K = w.shape
    assert K % 256 == 0
    out = np.empty((O, K // 256 * Q5K_BLOCK), dtype=np.uint8)
    lib().orc_quantize_q5_k(_ptr(w), O, K, _ptr(out))
    return out


def dequantize_q5_k(Wq: np.ndarray, K: int) -> np.ndarray:
    """uint8 [O][K/256*176] -> fp64 [O][K], every value d*sc*q - dmin*m exact."""
    Wq = np.ascontiguousarray(np.atleast_2d(Wq), dtype=np.uint8)
    assert K % 256 == 0 and Wq.shape[1] == K // 256 * Q5K_BLOCK
    out = np.empty((Wq.shape[0], K), dtype=np.float64)
    lib().orc_dequantize_q5_k(_ptr(Wq), Wq.shape[0], K, _ptr(out))
    return out


def q4_0_seg_row_bytes(K: int) -> int:
    """Bytes of one row in the Q4_0 segment layout (see oracle.c)."""
    assert K % 256 == 0 and K > 0
    return int(lib().orc_q4_0_seg_row_bytes(K))


def repack_q4_0_seg(Wq: np.ndarray, K: int) -> np.ndarray:
    """uint8 [O][K/32*18] Q4_0 rows -> uint8 [O][q4_0_seg_row_bytes(K)],
    the load-time segment layout (a byte rearrangement; see oracle.c)."""
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    assert K % 256 == 0 and Wq.shape[1] == K // QK * Q4_BLOCK
    O = Wq.shape[0]
    out = np.empty((O, q4_0_seg_row_bytes(K)), dtype=np.uint8)
    lib().orc_repack_q4_0_seg(_ptr(Wq), O, K, _ptr(out))
    return out


def rms_scale(x: np.ndarray, eps: float) -> float:
    x = np.ascontiguousarray(x, dtype=np.float32)
    return float(lib().orc_rms_scale(_ptr(x), x.shape[-1], float(np.float32(eps))))


def quantize_q8_0(x: np.ndarray, gamma: np.ndarray | None, eps: float = 1e-6,
                  add: np.ndarray | None = None) -> np.ndarray:
    """fp32 [N][K] (or [K]) -> uint8 [N][K/32*34] Q8_0 blocks; gamma=None = no
    norm; add = an fp32 addend applied after the norm and MUL: [K] (the same
    for every vector) or [N][K]."""
    x = np.ascontiguousarray(np.atleast_2d(x), dtype=np.float32)
    N, K = x.shape
    assert K % QK == 0
    g = None if gamma is None else np.ascontiguousarray(gamma, dtype=np.float32)
    out = np.empty((N, K // QK * Q8_BLOCK), dtype=np.uint8)
    if add is None:
        lib().orc_quantize_q8_0(_ptr(x), K, _ptr(g), float(np.float32(eps)), K, N, _ptr(out))
        return out
    a = np.ascontiguousarray(add, dtype=np.float32)
    if a.ndim == 1:
        assert a.shape[0] == K
        ldadd = 0
    else:
        assert a.shape == (N, K)
        ldadd = K
    lib().orc_quantize_q8_0_add(_ptr(x), K, _ptr(g), _ptr(a), ldadd, float(np.float32(eps)), K, N, _ptr(out))
    return out


def block_sums(Wq: np.ndarray, xq: np.ndarray, K: int, wtype: str = "q4_0") -> np.ndarray:
    """int32 [N][O][K/32] exact block sums; wtype "q4_0" (Q4_0 weights,
    sum (q-8) qx), "q8_0" (Q8_0 weights), "q4_k" or "q5_k" (k-quant weights,
    sum q qx per 32-weight sub-block)."""
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    xq = np.ascontiguousarray(np.atleast_2d(xq), dtype=np.uint8)
    O = Wq.shape[0]
    N = xq.shape[0]
    assert Wq.shape[1] == K // QK * _BYTES_PER_32[wtype]
    out = np.empty((N, O, K // QK), dtype=np.int32)
    fn = {"q4_0": lib().orc_block_sums, "q8_0": lib().orc_block_sums_q8w, "q4_k": lib().orc_block_sums_q4k,
          "q5_k": lib().orc_block_sums_q5k}[wtype]
    fn(_ptr(Wq), _ptr(xq), O, K, N, _ptr(out))
    return out


def matvec(Wq: np.ndarray, xq: np.ndarray, K: int, rows: np.ndarray | None = None,
           threads: int = 1, wtype: str = "q4_0"):
    """Reference y for N vectors: returns (y32 [N][R], y64 [N][R], S [N][R]).

    ``rows`` restricts the evaluation to the given row indices of Wq (R of
    them); otherwise all O rows.  ``threads`` > 1 splits rows over Python
    threads (the C call releases the GIL); results do not depend on it.
    ``wtype`` "q4_0" (Q4_0 weights), "q8_0" (Q8_0 weights), "q4_k" (Q4_K) or "q5_k" (Q5_K).
    """
    Wq = np.ascontiguousarray(Wq, dtype=np.uint8)
    xq = np.ascontiguousarray(np.atleast_2d(xq), dtype=np.uint8)
    O = Wq.shape[0]
    N = xq.shape[0]
    if rows is None:
        rows = np.arange(O, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    R = rows.shape[0]
    y32 = np.empty((N, R), dtype=np.float32)
    y64 = np.empty((N, R), dtype=np.float64)
    S = np.empty((N, R), dtype=np.float64)
    L = lib()
    assert Wq.shape[1] == K // QK * _BYTES_PER_32[wtype]
    mv = {"q4_0": L.orc_matvec, "q8_0": L.orc_matvec_q8w, "q4_k": L.orc_matvec_q4k, "q5_k": L.orc_matvec_q5k}[wtype]

    def run(lo, hi):
        if hi <= lo:
            return
        sub = np.ascontiguousarray(rows[lo:hi])
        a = np.empty((N, hi - lo), dtype=np.float32)
        b = np.empty((N, hi - lo), dtype=np.float64)
        c = np.empty((N, hi - lo), dtype=np.float64)
        mv(_ptr(Wq), _ptr(xq), O, K, N, _ptr(sub), hi - lo, _ptr(a), _ptr(b), _ptr(c))
        y32[:, lo:hi] = a
        y64[:, lo:hi] = b
        S[:, lo:hi] = c

    if threads <= 1 or R < 2 * threads:
        run(0, R)
    else:
        bounds = np.linspace(0, R, threads + 1).astype(np.int64)
        ts = [threading.Thread(target=run, args=(int(bounds[i]), int(bounds[i + 1])))
              for i in range(threads)]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
    return y32, y64, S
