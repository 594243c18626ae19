"""Python binding of the C ABI in include/qdg.h (ctypes; argument marshalling only).

Every function here has the name of the C entry point it calls, takes torch
tensors for the device buffers (PyTorch is only the allocator and the stream
provider) and raises ``QdgError`` when the library returns a negative status.
All arithmetic happens in the CUDA kernels of ``libqdg.so``; there is no other
code path, and importing this module fails loudly if the library cannot be
built or loaded.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

QK = 32
Q4_BLOCK = 18
Q8_BLOCK = 34

QDG_OK = 0
QDG_EINVAL = -1
QDG_EALIGN = -2
QDG_ESHAPE = -3
QDG_ECUDA = -4
QDG_ETIMEOUT = -5
QDG_EOVERFLOW = -6
QDG_OPT_PDL = 1

_lock = threading.Lock()
_lib = None


class QdgError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: status {status} ({status_string(status)})")


def lib() -> ctypes.CDLL:
    """Load libqdg.so (building it in-tree with nvcc when missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ctypes.CDLL(path, mode=ctypes.RTLD_GLOBAL)
            i64, p, f32, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
            sig = {
                "qnorm_quantize_q8_0": ([p, i64, p, f32, i64, i64, p, p], i32),
                "qnorm_add_quantize_q8_0": ([p, i64, p, p, i64, f32, i64, i64, p, p], i32),
                "q4_0_q8_0_gemv": ([p, p, p, i64, i64, p], i32),
                "q4_0_q8_0_gemv_group": ([p, p, p, i32, p, i64, p], i32),
                "q4_0_gemv_rmsnorm": ([p, p, p, f32, p, i64, i64, p, p], i32),
                "q4_0_gemv_rmsnorm_group": ([p, p, p, i32, p, p, f32, i64, p, p], i32),
                "q4_0_q8_0_gemm_small_n": ([p, p, p, i64, i64, i64, i64, p], i32),
                "quantize_q4_0": ([p, i64, i64, i64, p, p], i32),
                "qdg_device_status": ([p], i32),
                "qdg_status_string": ([i32], ctypes.c_char_p),
                "qdg_set_option": ([i32, i64], i32),
                "qdg_launch_count": ([i32], i64),
                "qdg_debug_block_sums": ([p, p, p, i64, i64, i64, i32, p], i32),
                "qdg_debug_timeout_probe": ([p], i32),
            }
            sig["q4_0_q8_0_gemm"] = ([p, p, p, i64, i64, i64, i64, p, i64, p], i32)
            sig["q4_0_q8_0_gemm_workspace_bytes"] = ([i64, i64], i64)
            sig["q4_0_q8_0_gemm_workspace_size"] = ([i64, i64, i64], i64)
            sig["q4_0_q8_0_gemm_static"] = ([p, p, p, i64, i64, i64, i64, p], i32)
            sig["q8_0_q8_0_gemv"] = ([p, p, p, i64, i64, p], i32)
            sig["q8_0_q8_0_gemv_group"] = ([p, p, p, i32, p, i64, p], i32)
            sig["q4_k_q8_0_gemv"] = ([p, p, p, i64, i64, p], i32)
            sig["quantize_q4_k"] = ([p, i64, i64, i64, p, p], i32)
            sig["q4_k_q8_0_gemv_group"] = ([p, p, p, i32, p, i64, p], i32)
            sig["q5_k_q8_0_gemv"] = ([p, p, p, i64, i64, p], i32)
            sig["quantize_q5_k"] = ([p, i64, i64, i64, p, p], i32)
            sig["q5_k_q8_0_gemv_group"] = ([p, p, p, i32, p, i64, p], i32)
            sig["q4_0s_gemv_rmsnorm_group"] = ([p, p, p, i32, p, p, f32, i64, p, p], i32)
            sig["q4_0s_q8_0_gemm_small_n"] = ([p, p, p, i64, i64, i64, i64, p], i32)
            sig["q4_0_seg_row_bytes"] = ([i64], i64)
            sig["q4_0_repack_seg"] = ([p, p, i64, i64, p], i32)
            sig["q4_0s_q8_0_gemv"] = ([p, p, p, i64, i64, p], i32)
            sig["q4_0s_q8_0_gemv_group"] = ([p, p, p, i32, p, i64, p], i32)
            sig["qdg_stage_copy"] = ([p, p, i64, p], i32)
            sig["q4_0s_gemv_chain_workspace_bytes"] = ([], i64)
            sig["q4_0s_gemv_chain"] = ([p, i32, f32, p, p], i32)
            for name, (args, res) in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def library_path() -> str:
    return _build.LIB


def status_string(status: int) -> str:
    try:
        return lib().qdg_status_string(int(status)).decode()
    except OSError:
        return "unknown"


def _check(status: int, what: str) -> None:
    if status != QDG_OK:
        raise QdgError(status, what)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def q4_0_nbytes(O: int, K: int) -> int:
    return O * (K // QK) * Q4_BLOCK


def q8_0_nbytes(N: int, K: int) -> int:
    return N * (K // QK) * Q8_BLOCK


# ------------------------------------------------------------------ entry points
def qnorm_quantize_q8_0(x, gamma, eps: float, xq, K: int | None = None, N: int | None = None,
                        ldx: int | None = None, stream=None) -> None:
    """Fused RMSNorm*gamma -> Q8_0 (gamma=None: plain Q8_0).  x fp32 [N][ldx]."""
    if K is None:
        K = x.shape[-1]
    if N is None:
        N = 1 if x.dim() == 1 else x.shape[0]
    if ldx is None:
        ldx = K if x.dim() == 1 else x.stride(0)
    _check(lib().qnorm_quantize_q8_0(_ptr(x), ldx, _ptr(gamma), float(eps), K, N, _ptr(xq), _stream(stream)),
           "qnorm_quantize_q8_0")



def qnorm_add_quantize_q8_0(x, gamma, add, eps: float, xq, K: int | None = None, N: int | None = None,
                            ldx: int | None = None, ldadd: int | None = None, stream=None) -> None:
    """Fused RMSNorm*gamma + add -> Q8_0.  add fp32 [K] (broadcast, ldadd 0) or [N][ldadd]."""
    if K is None:
        K = x.shape[-1]
    if N is None:
        N = 1 if x.dim() == 1 else x.shape[0]
    if ldx is None:
        ldx = K if x.dim() == 1 else x.stride(0)
    if ldadd is None:
        ldadd = 0 if add.dim() == 1 else add.stride(0)
    _check(lib().qnorm_add_quantize_q8_0(_ptr(x), ldx, _ptr(gamma), _ptr(add), ldadd, float(eps), K, N, _ptr(xq),
                                         _stream(stream)), "qnorm_add_quantize_q8_0")

def q4_0_q8_0_gemv(W, xq, y, O: int, K: int, stream=None) -> None:
    _check(lib().q4_0_q8_0_gemv(_ptr(W), _ptr(xq), _ptr(y), O, K, _stream(stream)), "q4_0_q8_0_gemv")


def q4_0_q8_0_gemv_group(Ws, ys, Os, xq, K: int, stream=None) -> None:
    """GEMV for up to 4 matrices sharing one Q8_0 vector (one launch)."""
    n = len(Ws)
    W_arr = (ctypes.c_void_p * n)(*[_ptr(w) for w in Ws])
    y_arr = (ctypes.c_void_p * n)(*[_ptr(t) for t in ys])
    O_arr = (ctypes.c_int64 * n)(*[int(o) for o in Os])
    _check(lib().q4_0_q8_0_gemv_group(W_arr, y_arr, O_arr, n, _ptr(xq), K, _stream(stream)), "q4_0_q8_0_gemv_group")


def q8_0_q8_0_gemv(W, xq, y, O: int, K: int, stream=None) -> None:
    """y = W * x with Q8_0 weights."""
    _check(lib().q8_0_q8_0_gemv(_ptr(W), _ptr(xq), _ptr(y), O, K, _stream(stream)), "q8_0_q8_0_gemv")


def q8_0_q8_0_gemv_group(Ws, ys, Os, xq, K: int, stream=None) -> None:
    """Q8_0-weight GEMV for up to 4 matrices sharing one Q8_0 vector (one launch)."""
    n = len(Ws)
    W_arr = (ctypes.c_void_p * n)(*[_ptr(w) for w in Ws])
    y_arr = (ctypes.c_void_p * n)(*[_ptr(t) for t in ys])
    O_arr = (ctypes.c_int64 * n)(*[int(o) for o in Os])
    _check(lib().q8_0_q8_0_gemv_group(W_arr, y_arr, O_arr, n, _ptr(xq), K, _stream(stream)), "q8_0_q8_0_gemv_group")


def quantize_q4_k(w, Wq, O: int | None = None, K: int | None = None, ldw: int | None = None,
                  stream=None) -> None:
    """fp32 [O][K] weights -> Q4_K super-blocks (load-time preparation)."""
    if O is None:
        O, K = w.shape
    ldw = K if ldw is None else ldw
    _check(lib().quantize_q4_k(_ptr(w), ldw, O, K, _ptr(Wq), _stream(stream)), "quantize_q4_k")


def q4_k_q8_0_gemv(W, xq, y, O: int, K: int, stream=None) -> None:
    """y = W * x with Q4_K weights (256-weight super-blocks, see include/qdg.h)."""
    _check(lib().q4_k_q8_0_gemv(_ptr(W), _ptr(xq), _ptr(y), O, K, _stream(stream)), "q4_k_q8_0_gemv")


def q4_k_q8_0_gemv_group(Ws, ys, Os, xq, K: int, stream=None) -> None:
    n = len(Ws)
    W_arr = (ctypes.c_void_p * n)(*[_ptr(w) for w in Ws])
    y_arr = (ctypes.c_void_p * n)(*[_ptr(t) for t in ys])
    O_arr = (ctypes.c_int64 * n)(*[int(o) for o in Os])
    _check(lib().q4_k_q8_0_gemv_group(W_arr, y_arr, O_arr, n, _ptr(xq), K, _stream(stream)), "q4_k_q8_0_gemv_group")


def quantize_q5_k(w, Wq, O: int | None = None, K: int | None = None, ldw: int | None = None,
                  stream=None) -> None:
    """fp32 [O][K] weights -> Q5_K super-blocks (load-time preparation)."""
    if O is None:
        O, K = w.shape
    ldw = K if ldw is None else ldw
    _check(lib().quantize_q5_k(_ptr(w), ldw, O, K, _ptr(Wq), _stream(stream)), "quantize_q5_k")


def q5_k_q8_0_gemv(W, xq, y, O: int, K: int, stream=None) -> None:
    """y = W * x with Q5_K weights (256-weight super-blocks, see include/qdg.h)."""
    _check(lib().q5_k_q8_0_gemv(_ptr(W), _ptr(xq), _ptr(y), O, K, _stream(stream)), "q5_k_q8_0_gemv")


def q5_k_q8_0_gemv_group(Ws, ys, Os, xq, K: int, stream=None) -> None:
    n = len(Ws)
    W_arr = (ctypes.c_void_p * n)(*[_ptr(w) for w in Ws])
    y_arr = (ctypes.c_void_p * n)(*[_ptr(t) for t in ys])
    O_arr = (ctypes.c_int64 * n)(*[int(o) for o in Os])
    _check(lib().q5_k_q8_0_gemv_group(W_arr, y_arr, O_arr, n, _ptr(xq), K, _stream(stream)), "q5_k_q8_0_gemv_group")


def q4_0_seg_row_bytes(K: int) -> int:
    """Bytes of one row of K weights in the segment layout."""
    r = int(lib().q4_0_seg_row_bytes(K))
    _check(min(r, 0), "q4_0_seg_row_bytes")
    return r


def q4_0_seg_nbytes(O: int, K: int) -> int:
    return O * q4_0_seg_row_bytes(K)


def q4_0_repack_seg(W, Wr, O: int, K: int, stream=None) -> None:
    """Q4_0 rows -> segment layout (load time, bit-exact rearrangement)."""
    _check(lib().q4_0_repack_seg(_ptr(W), _ptr(Wr), O, K, _stream(stream)), "q4_0_repack_seg")


def qdg_stage_copy(dst, src, nbytes: int | None = None, stream=None) -> None:
    """Kernel copy between device memory and mapped pinned host memory (a
    step's inputs in, its outputs out); nbytes defaults to src's size."""
    if nbytes is None:
        nbytes = src.numel() * src.element_size()
    _check(lib().qdg_stage_copy(_ptr(dst), _ptr(src), int(nbytes), _stream(stream)), "qdg_stage_copy")


def q4_0s_q8_0_gemv(Wr, xq, y, O: int, K: int, stream=None) -> None:
    """y = W * x with W in the segment layout."""
    _check(lib().q4_0s_q8_0_gemv(_ptr(Wr), _ptr(xq), _ptr(y), O, K, _stream(stream)), "q4_0s_q8_0_gemv")


def q4_0s_q8_0_gemv_group(Ws, ys, Os, xq, K: int, stream=None) -> None:
    """Segment-layout GEMV for up to 4 matrices sharing one Q8_0 vector."""
    n = len(Ws)
    W_arr = (ctypes.c_void_p * n)(*[_ptr(w) for w in Ws])
    y_arr = (ctypes.c_void_p * n)(*[_ptr(t) for t in ys])
    O_arr = (ctypes.c_int64 * n)(*[int(o) for o in Os])
    _check(lib().q4_0s_q8_0_gemv_group(W_arr, y_arr, O_arr, n, _ptr(xq), K, _stream(stream)),
           "q4_0s_q8_0_gemv_group")


def q4_0_gemv_rmsnorm(W, x, gamma, eps: float, y, O: int, K: int, xq_out=None, stream=None) -> None:
    """Fused RMSNorm*gamma -> Q8_0 -> GEMV (gamma=None: plain quantization)."""
    _check(lib().q4_0_gemv_rmsnorm(_ptr(W), _ptr(x), _ptr(gamma), float(eps), _ptr(y), O, K, _ptr(xq_out),
                                   _stream(stream)), "q4_0_gemv_rmsnorm")


def q4_0_gemv_rmsnorm_group(Ws, ys, Os, x, gamma, eps: float, K: int, xq_out=None, stream=None) -> None:
    """Fused route for up to 4 matrices sharing the input x (one launch)."""
    n = len(Ws)
    W_arr = (ctypes.c_void_p * n)(*[_ptr(w) for w in Ws])
    y_arr = (ctypes.c_void_p * n)(*[_ptr(t) for t in ys])
    O_arr = (ctypes.c_int64 * n)(*[int(o) for o in Os])
    _check(lib().q4_0_gemv_rmsnorm_group(W_arr, y_arr, O_arr, n, _ptr(x), _ptr(gamma), float(eps), K,
                                         _ptr(xq_out), _stream(stream)), "q4_0_gemv_rmsnorm_group")


def q4_0s_gemv_rmsnorm_group(Ws, ys, Os, x, gamma, eps: float, K: int, xq_out=None, stream=None) -> None:
    """Fused route on the segment layout for up to 4 matrices sharing the input x."""
    n = len(Ws)
    W_arr = (ctypes.c_void_p * n)(*[_ptr(w) for w in Ws])
    y_arr = (ctypes.c_void_p * n)(*[_ptr(t) for t in ys])
    O_arr = (ctypes.c_int64 * n)(*[int(o) for o in Os])
    _check(lib().q4_0s_gemv_rmsnorm_group(W_arr, y_arr, O_arr, n, _ptr(x), _ptr(gamma), float(eps), K,
                                          _ptr(xq_out), _stream(stream)), "q4_0s_gemv_rmsnorm_group")


class ChainStage(ctypes.Structure):
    """qdg_chain_stage of include/qdg.h."""
    _fields_ = [("x", ctypes.c_void_p), ("gamma", ctypes.c_void_p), ("xq_out", ctypes.c_void_p),
                ("K", ctypes.c_int64), ("count", ctypes.c_int),
                ("W", ctypes.c_void_p * 4), ("y", ctypes.c_void_p * 4), ("O", ctypes.c_int64 * 4)]


def q4_0s_gemv_chain_workspace_bytes() -> int:
    return int(lib().q4_0s_gemv_chain_workspace_bytes())


def chain_stages(stages):
    """Marshal stage descriptions -- dicts with x, gamma (or None), K, Ws, ys,
    Os and optionally xq_out -- into the C array the chain call takes."""
    arr = (ChainStage * len(stages))()
    for d, st in zip(arr, stages):
        d.x = _ptr(st["x"])
        d.gamma = _ptr(st.get("gamma"))
        d.xq_out = _ptr(st.get("xq_out"))
        d.K = int(st["K"])
        n = len(st["Ws"])
        d.count = n
        for i in range(min(n, 4)):
            d.W[i] = _ptr(st["Ws"][i])
            d.y[i] = _ptr(st["ys"][i])
            d.O[i] = int(st["Os"][i])
    return arr


def q4_0s_gemv_chain(stages, eps: float, workspace, stream=None) -> None:
    """A decode step's stages (norm/quantize + grouped segment-layout GEMV each)
    in one launch; ``stages`` as for chain_stages(), or its result."""
    arr = stages if isinstance(stages, ctypes.Array) else chain_stages(stages)
    _check(lib().q4_0s_gemv_chain(arr, len(arr), float(eps), _ptr(workspace), _stream(stream)), "q4_0s_gemv_chain")


def q4_0s_q8_0_gemm_small_n(Wr, xq, y, ldy: int, O: int, K: int, N: int, stream=None) -> None:
    """Small-N product on the segment layout, N = 1..8."""
    _check(lib().q4_0s_q8_0_gemm_small_n(_ptr(Wr), _ptr(xq), _ptr(y), ldy, O, K, N, _stream(stream)),
           "q4_0s_q8_0_gemm_small_n")


def q4_0_q8_0_gemm_small_n(W, xq, y, ldy: int, O: int, K: int, N: int, stream=None) -> None:
    _check(lib().q4_0_q8_0_gemm_small_n(_ptr(W), _ptr(xq), _ptr(y), ldy, O, K, N, _stream(stream)),
           "q4_0_q8_0_gemm_small_n")


def q4_0_q8_0_gemm_workspace_size(O: int, K: int, T: int) -> int:
    n = int(lib().q4_0_q8_0_gemm_workspace_size(O, K, T))
    if n < 0:
        raise QdgError(n, "q4_0_q8_0_gemm_workspace_size")
    return n


def q4_0_q8_0_gemm_workspace_bytes(K: int, T: int) -> int:
    n = int(lib().q4_0_q8_0_gemm_workspace_bytes(K, T))
    if n < 0:
        raise QdgError(n, "q4_0_q8_0_gemm_workspace_bytes")
    return n


def q4_0_q8_0_gemm(W, xq, y, ldy: int, O: int, K: int, T: int, workspace, workspace_bytes: int | None = None,
                   stream=None) -> None:
    """Prefill product; `workspace` is caller-owned device memory of at least
    q4_0_q8_0_gemm_workspace_bytes(K, T) bytes (a uint8 tensor: its size is
    used when workspace_bytes is None)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0
    _check(lib().q4_0_q8_0_gemm(_ptr(W), _ptr(xq), _ptr(y), ldy, O, K, T, _ptr(workspace), workspace_bytes,
                                _stream(stream)), "q4_0_q8_0_gemm")


def q4_0_q8_0_gemm_static(W, xq, y, ldy: int, O: int, K: int, T: int, stream=None) -> None:
    """Prefill product with the library's own fixed-size scratch (no allocation)."""
    _check(lib().q4_0_q8_0_gemm_static(_ptr(W), _ptr(xq), _ptr(y), ldy, O, K, T, _stream(stream)),
           "q4_0_q8_0_gemm_static")


def quantize_q4_0(w, Wq, O: int | None = None, K: int | None = None, ldw: int | None = None,
                  stream=None) -> None:
    if O is None:
        O, K = w.shape
    if ldw is None:
        ldw = w.stride(0) if w.dim() == 2 else K
    _check(lib().quantize_q4_0(_ptr(w), ldw, O, K, _ptr(Wq), _stream(stream)), "quantize_q4_0")


def qdg_device_status(stream=None) -> int:
    return int(lib().qdg_device_status(_stream(stream)))


def qdg_set_option(option: int, value: int) -> None:
    _check(lib().qdg_set_option(option, value), "qdg_set_option")


def qdg_launch_count(which: int = -1) -> int:
    return int(lib().qdg_launch_count(which))


def qdg_debug_block_sums(W, xq, isum, O: int, K: int, N: int, path: int, stream=None) -> None:
    _check(lib().qdg_debug_block_sums(_ptr(W), _ptr(xq), _ptr(isum), O, K, N, path, _stream(stream)),
           "qdg_debug_block_sums")


def qdg_debug_timeout_probe(stream=None) -> None:
    _check(lib().qdg_debug_timeout_probe(_stream(stream)), "qdg_debug_timeout_probe")
