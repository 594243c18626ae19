"""The C ABI without a GPU: the library builds, loads, exports every symbol
include/qdg.h declares, and rejects bad arguments on the host before any
CUDA call (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qdg.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"QDG_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    from quantized_decode_gemv_rms_gb300 import qdg
    return qdg.lib()


def test_header_declares_entry_points():
    names = declared_symbols()
    for must in ("qnorm_quantize_q8_0", "qnorm_add_quantize_q8_0", "q4_0_q8_0_gemv", "q4_0_q8_0_gemm_small_n", "q4_0_q8_0_gemm",
                 "q4_0_q8_0_gemm_workspace_bytes", "q4_0_q8_0_gemm_workspace_size", "qdg_stage_copy", "quantize_q4_0", "q4_0_repack_seg", "q4_0s_q8_0_gemv",
                 "q4_0s_q8_0_gemv_group", "q4_0s_gemv_rmsnorm_group", "q4_0s_q8_0_gemm_small_n", "q4_0_seg_row_bytes", "q8_0_q8_0_gemv", "q8_0_q8_0_gemv_group",
                 "q4_0s_gemv_chain", "q4_0s_gemv_chain_workspace_bytes", "qdg_device_status", "qdg_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), f"libqdg.so does not export {name}"


def test_status_strings(L):
    from quantized_decode_gemv_rms_gb300 import qdg
    for code in (qdg.QDG_OK, qdg.QDG_EINVAL, qdg.QDG_EALIGN, qdg.QDG_ESHAPE, qdg.QDG_ECUDA,
                 qdg.QDG_ETIMEOUT, qdg.QDG_EOVERFLOW):
        assert qdg.status_string(code) not in ("", "unknown status")
    assert qdg.status_string(12345) == "unknown status"


A16 = 0x10000          # fake, 16-byte aligned device addresses: never dereferenced on the host
A2 = 0x10002           # 2-byte aligned only


def test_qnorm_host_validation(L):
    f = L.qnorm_quantize_q8_0
    assert f(None, 256, None, 1e-6, 256, 1, A16, None) == -1          # null x
    assert f(A16, 256, None, 1e-6, 256, 1, None, None) == -1          # null xq
    assert f(A16, 256, None, 1e-6, 0, 1, A16, None) == -1             # K = 0
    assert f(A16, 256, None, 1e-6, 256, 0, A16, None) == -1           # N = 0
    assert f(A16, 100, None, 1e-6, 256, 1, A16, None) == -1           # ldx < K
    assert f(A16, 256, None, -1.0, 256, 1, A16, None) == -1           # eps < 0
    assert f(A16, 256, None, float("nan"), 256, 1, A16, None) == -1   # eps NaN
    assert f(A16, 48, None, 1e-6, 48, 1, A16, None) == -3             # K % 32
    assert f(A2, 256, None, 1e-6, 256, 1, A16, None) == -2            # x misaligned
    assert f(A16, 256, A2, 1e-6, 256, 1, A16, None) == -2             # gamma misaligned
    assert f(A16, 256, None, 1e-6, 256, 1, A16 + 1, None) == -2       # xq misaligned


def test_qnorm_add_host_validation(L):
    f = L.qnorm_add_quantize_q8_0
    assert f(A16, 256, A16, None, 0, 1e-6, 256, 1, A16, None) == -1     # null addend
    assert f(A16, 256, A16, A16, 100, 1e-6, 256, 2, A16, None) == -1    # 0 < ldadd < K
    assert f(A16, 256, A16, A2 + 1, 0, 1e-6, 256, 1, A16, None) == -2   # addend misaligned
    assert f(A16, 256, A16, A16, 0, 1e-6, 48, 1, A16, None) == -3       # K % 32


def test_gemv_host_validation(L):
    f = L.q4_0_q8_0_gemv
    assert f(None, A16, A16, 8, 256, None) == -1
    assert f(A16, A16, None, 8, 256, None) == -1
    assert f(A16, A16, A16, 0, 256, None) == -1
    assert f(A16, A16, A16, 8, 128, None) == -3       # K % 256
    assert f(A16, A16, A16, 8, 65536, None) == -3     # K beyond the maximum
    assert f(A2, A16, A16, 8, 256, None) == -2        # W not 16-byte aligned
    assert f(A16, A2, A16, 8, 256, None) == -2        # xq not 4-byte aligned


def test_q8w_gemv_host_validation(L):
    f = L.q8_0_q8_0_gemv
    assert f(None, A16, A16, 8, 256, None) == -1
    assert f(A16, A16, None, 8, 256, None) == -1
    assert f(A16, A16, A16, 0, 256, None) == -1
    assert f(A16, A16, A16, 8, 128, None) == -3       # K % 256
    assert f(A16, A16, A16, 8, 65536, None) == -3     # K beyond the maximum
    assert f(A2, A16, A16, 8, 256, None) == -2        # W not 16-byte aligned
    assert f(A16, A2, A16, 8, 256, None) == -2        # xq not 4-byte aligned
    g = L.q8_0_q8_0_gemv_group
    W = (ctypes.c_void_p * 5)(*([A16] * 5))
    Y = (ctypes.c_void_p * 5)(*([A16] * 5))
    O = (ctypes.c_int64 * 5)(*([8] * 5))
    assert g(W, Y, O, 5, A16, 256, None) == -1
    assert g(W, None, O, 2, A16, 256, None) == -1


def test_seg_layout_host_validation(L):
    import oracle
    for K in (256, 2304, 4096, 4352, 14336, 32768):
        assert L.q4_0_seg_row_bytes(K) == oracle.q4_0_seg_row_bytes(K)
    assert L.q4_0_seg_row_bytes(0) == -1
    assert L.q4_0_seg_row_bytes(128) == -3
    assert L.q4_0_seg_row_bytes(65536) == -3
    r = L.q4_0_repack_seg
    assert r(None, A16, 8, 256, None) == -1
    assert r(A16, None, 8, 256, None) == -1
    assert r(A16, A16, 0, 256, None) == -1
    assert r(A16, A16, 8, 96, None) == -3          # K % 256
    assert r(A16 + 1, A16, 8, 256, None) == -2     # W not 2-byte aligned
    assert r(A16, A2, 8, 256, None) == -2          # Wr not 16-byte aligned
    f = L.q4_0s_q8_0_gemv
    assert f(None, A16, A16, 8, 256, None) == -1
    assert f(A16, A16, None, 8, 256, None) == -1
    assert f(A16, A16, A16, 0, 256, None) == -1
    assert f(A16, A16, A16, 8, 128, None) == -3
    assert f(A16, A16, A16, 8, 65536, None) == -3
    assert f(A2, A16, A16, 8, 256, None) == -2     # Wr not 16-byte aligned
    assert f(A16, A16 + 1, A16, 8, 256, None) == -2  # xq not 2-byte aligned
    g = L.q4_0s_q8_0_gemv_group
    W = (ctypes.c_void_p * 5)(*([A16] * 5))
    Y = (ctypes.c_void_p * 5)(*([A16] * 5))
    O = (ctypes.c_int64 * 5)(*([8] * 5))
    assert g(W, Y, O, 5, A16, 256, None) == -1    # more than 4 matrices
    assert g(W, Y, O, 0, A16, 256, None) == -1


def test_fused_host_validation(L):
    f = L.q4_0_gemv_rmsnorm
    assert f(A16, None, None, 1e-6, A16, 8, 256, None, None) == -1      # null x
    assert f(A16, A16, None, -1.0, A16, 8, 256, None, None) == -1       # eps < 0
    assert f(A16, A16, None, 1e-6, A16, 8, 320, None, None) == -3       # K % 256
    assert f(A16, A16 + 4, None, 1e-6, A16, 8, 256, None, None) == -2   # x not 16-byte aligned
    assert f(A16, A16, A16 + 8, 1e-6, A16, 8, 256, None, None) == -2    # gamma not 16-byte aligned
    assert f(A16, A16, None, 1e-6, A16, 8, 256, A2, None) == -2         # xq_out not 4-byte aligned


def test_seg_small_n_host_validation(L):
    f = L.q4_0s_q8_0_gemm_small_n
    assert f(A16, A16, A16, 8, 8, 256, 9, None) == -1      # N = 9
    assert f(A16, A16, A16, 8, 8, 256, 0, None) == -1      # N = 0
    assert f(A16, A16, A16, 4, 8, 256, 3, None) == -1      # ldy < O (MMA path)
    assert f(A16, A16, A16, 8, 8, 384, 5, None) == -3      # K % 256 (MMA path)
    assert f(A16, A16 + 2, A16, 8, 8, 256, 8, None) == -2  # xq not 16-byte aligned (MMA path)
    assert f(A16, A16, None, 8, 8, 256, 2, None) == -1     # null y
    assert f(A16, A16, A16, 4, 8, 256, 2, None) == -1      # ldy < O
    assert f(A16, A16, A16, 8, 8, 384, 2, None) == -3      # K % 256
    assert f(A2, A16, A16, 8, 8, 256, 2, None) == -2       # Wr not 16-byte aligned
    assert f(A16, A16 + 1, A16, 8, 8, 256, 2, None) == -2  # xq not 2-byte aligned
    assert L.qdg_debug_block_sums(A16, A16, A16, 8, 256, 9, 5, None) == -1   # segment small-N: N <= 8


def test_fused_seg_host_validation(L):
    f = L.q4_0s_gemv_rmsnorm_group
    W = (ctypes.c_void_p * 2)(A16, A16)
    Y = (ctypes.c_void_p * 2)(A16, A16)
    O = (ctypes.c_int64 * 2)(8, 8)
    assert f(W, Y, O, 2, None, None, 1e-6, 256, None, None) == -1      # null x
    assert f(W, Y, O, 0, A16, None, 1e-6, 256, None, None) == -1       # count 0
    assert f(W, Y, O, 2, A16, None, -1.0, 256, None, None) == -1       # eps < 0
    assert f(W, Y, O, 2, A16, None, 1e-6, 320, None, None) == -3       # K % 256
    assert f(W, Y, O, 2, A16, None, 1e-6, 16640, None, None) == -3     # K beyond the fused maximum (16384)
    assert f(W, Y, O, 2, A16 + 4, None, 1e-6, 256, None, None) == -2   # x not 16-byte aligned
    assert f(W, Y, O, 2, A16, A16 + 8, 1e-6, 256, None, None) == -2    # gamma not 16-byte aligned
    assert f(W, Y, O, 2, A16, None, 1e-6, 256, A2, None) == -2         # xq_out not 4-byte aligned


def test_fused_group_host_validation(L):
    import ctypes
    f = L.q4_0_gemv_rmsnorm_group
    W = (ctypes.c_void_p * 2)(A16, A16)
    Y = (ctypes.c_void_p * 2)(A16, A16)
    O = (ctypes.c_int64 * 2)(8, 8)
    assert f(W, Y, O, 0, A16, None, 1e-6, 256, None, None) == -1        # count 0
    assert f(W, Y, O, 5, A16, None, 1e-6, 256, None, None) == -1        # count > 4
    assert f(W, Y, O, 2, A16, None, 1e-6, 320, None, None) == -3        # K % 256
    assert f(W, Y, O, 2, A16, None, 1e-6, 32768, None, None) == -3      # K beyond the fused maximum
    Wb = (ctypes.c_void_p * 2)(A16, A2)
    assert f(Wb, Y, O, 2, A16, None, 1e-6, 256, None, None) == -2       # second W misaligned
    Ob = (ctypes.c_int64 * 2)(8, 0)
    assert f(W, Y, Ob, 2, A16, None, 1e-6, 256, None, None) == -1       # empty matrix


def test_gemv_group_host_validation(L):
    import ctypes
    f = L.q4_0_q8_0_gemv_group
    W = (ctypes.c_void_p * 2)(A16, A16)
    Y = (ctypes.c_void_p * 2)(A16, A16)
    O = (ctypes.c_int64 * 2)(8, 8)
    assert f(W, Y, O, 0, A16, 256, None) == -1          # count 0
    assert f(W, Y, O, 5, A16, 256, None) == -1          # count > 4
    assert f(W, None, O, 2, A16, 256, None) == -1       # no outputs
    assert f(W, Y, O, 2, A16, 384, None) == -3          # K % 256
    assert f(W, Y, O, 2, A2, 256, None) == -2           # xq not 4-byte aligned
    Ob = (ctypes.c_int64 * 2)(8, -1)
    assert f(W, Y, Ob, 2, A16, 256, None) == -1         # negative rows


def test_small_n_host_validation(L):
    f = L.q4_0_q8_0_gemm_small_n
    assert f(A16, A16, A16, 8, 8, 256, 0, None) == -1      # N = 0
    assert f(A16, A16, A16, 8, 8, 256, 9, None) == -1      # N > 8
    assert f(A16, A16, A16, 4, 8, 256, 2, None) == -1      # ldy < O
    assert f(A16, A16, None, 8, 8, 256, 2, None) == -1
    assert f(A16, A16, A16, 8, 8, 384, 2, None) == -3      # K % 256
    assert f(A16, A2, A16, 8, 8, 256, 2, None) == -2       # xq must be 16-byte aligned
    assert f(A16, A16, A16, 8, 8, 32768 + 256, 2, None) == -3   # K beyond the maximum


def test_gemm_host_validation(L):
    f = L.q4_0_q8_0_gemm
    need = L.q4_0_q8_0_gemm_workspace_bytes(256, 4)
    assert need == 1 * 8 * 8704                                      # one token tile, 8 blocks
    assert L.q4_0_q8_0_gemm_workspace_bytes(256, 129) == 2 * 8 * 8704
    assert L.q4_0_q8_0_gemm_workspace_bytes(320, 4) == -3             # K % 256
    assert L.q4_0_q8_0_gemm_workspace_bytes(256, 0) == -1
    assert L.q4_0_q8_0_gemm_workspace_size(14336, 256, 129) == 2 * 8 * 8704   # O does not change it
    assert L.q4_0_q8_0_gemm_workspace_size(0, 256, 129) == -1
    assert L.q4_0_q8_0_gemm_workspace_size((1 << 30) + 1, 256, 129) == -3   # the product refuses this O
    assert f(A16, A16, None, 8, 8, 256, 4, A16, need, None) == -1     # null y
    assert f(A16, A16, A16, 4, 8, 256, 4, A16, need, None) == -1      # ldy < O
    assert f(A16, A16, A16, 8, 8, 256, 0, A16, need, None) == -1      # T = 0
    assert f(A16, A16, A16, 8, 8, 320, 4, A16, need, None) == -3      # K % 256
    assert f(A2, A16, A16, 8, 8, 256, 4, A16, need, None) == -2       # W misaligned
    assert f(A16, A2, A16, 8, 8, 256, 4, A16, need, None) == -2       # xq misaligned
    assert f(A16, A16, A16, 8, 8, 256, 4, None, need, None) == -1     # no workspace
    assert f(A16, A16, A16, 8, 8, 256, 4, A16, need - 16, None) == -1 # workspace too small
    assert f(A16, A16, A16, 8, 8, 256, 4, A2, need, None) == -2       # workspace misaligned


def test_quantize_q4_0_host_validation(L):
    f = L.quantize_q4_0
    assert f(None, 32, 1, 32, A16, None) == -1
    assert f(A16, 16, 1, 32, A16, None) == -1               # ldw < K
    assert f(A16, 40, 1, 40, A16, None) == -3               # K % 32
    assert f(A2 + 1, 32, 1, 32, A16, None) == -2


def test_stage_copy_rejects_bad_arguments(L):
    f = L.qdg_stage_copy
    assert f(None, A16, 16, None) == -1
    assert f(A16, None, 16, None) == -1
    assert f(A16, A16, -16, None) == -1
    assert f(A16, A16, 0, None) == 0                     # nothing to do, nothing launched
    assert f(A16 + 8, A16, 16, None) == -2
    assert f(A16, A16 + 4, 16, None) == -2
    assert f(A16, A16, 24, None) == -2                   # size not a multiple of 16


def test_options_and_counters(L):
    assert L.qdg_set_option(99, 1) == -1
    assert L.qdg_set_option(1, 2) == -1
    assert L.qdg_set_option(1, 0) == 0
    assert L.qdg_launch_count(-1) >= 0
    assert L.qdg_launch_count(14) >= 0
    assert L.qdg_launch_count(15) == -1
    assert L.qdg_launch_count(10) >= 0
    assert L.qdg_debug_block_sums(A16, A16, None, 8, 256, 1, 0, None) == -1
    assert L.qdg_debug_block_sums(A16, A16, A16, 8, 256, 1, 9, None) == -1
    assert L.qdg_debug_block_sums(A16, A16, A16, 8, 256, 2, 0, None) == -1   # gemv path needs N == 1
    assert L.qdg_debug_block_sums(A16, A16, A16, 8, 256, 2, 3, None) == -1   # so does the segment-layout gemv
    assert L.qdg_debug_block_sums(A16, A16, A16, 8, 256, 2, 4, None) == -1   # and the Q8_0-weight gemv


def test_binding_names_match_header():
    from quantized_decode_gemv_rms_gb300 import qdg
    for name in declared_symbols():
        if name in ("qdg_status_string",):
            continue
        assert hasattr(qdg, name), f"binding lacks {name}"


def test_chain_host_validation(L):
    from quantized_decode_gemv_rms_gb300 import qdg
    assert L.q4_0s_gemv_chain_workspace_bytes() == 64 + 512 * 40

    def stage(K=4096, count=1, x=A16, gamma=None, W=A16, y=A16, O=8):
        st = (qdg.ChainStage * 1)()
        st[0].x, st[0].gamma, st[0].K, st[0].count = x, gamma, K, count
        for i in range(4):
            st[0].W[i], st[0].y[i], st[0].O[i] = W, y, O
        return st

    f = L.q4_0s_gemv_chain
    two = (qdg.ChainStage * 9)()
    assert f(stage(), 0, 1e-6, A16, None) == -1                   # no stage
    assert f(two, 9, 1e-6, A16, None) == -1                       # more than eight stages
    assert f(stage(), 1, 1e-6, None, None) == -1                  # no workspace
    assert f(stage(), 1, -1.0, A16, None) == -1                   # eps < 0
    assert f(stage(), 1, 1e-6, A2, None) == -2                    # workspace not 16-byte aligned
    assert f(stage(count=0), 1, 1e-6, A16, None) == -1            # no matrix
    assert f(stage(count=5), 1, 1e-6, A16, None) == -1            # more than four matrices
    assert f(stage(x=None), 1, 1e-6, A16, None) == -1             # null x
    assert f(stage(K=320), 1, 1e-6, A16, None) == -3              # K % 256
    assert f(stage(K=16384 + 256), 1, 1e-6, A16, None) == -3      # K beyond the maximum
    assert f(stage(x=A2), 1, 1e-6, A16, None) == -2               # x must be 16-byte aligned
    assert f(stage(gamma=A2), 1, 1e-6, A16, None) == -2           # gamma likewise
    assert f(stage(W=A2), 1, 1e-6, A16, None) == -2               # weights 16-byte aligned
    assert f(stage(O=0), 1, 1e-6, A16, None) == -1                # no rows
    assert f(stage(W=None), 1, 1e-6, A16, None) == -1             # null weights
