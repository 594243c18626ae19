"""GPU parity: fused RMSNorm*gamma -> Q8_0 and the Q4_0 weight quantizer
against the CPU oracle, byte for byte (codes and fp16 scale bits)."""
import numpy as np
import pytest

import oracle
from quantized_decode_gemv_rms_gb300 import qdg, synth
from helpers import empty_u8, to_dev, to_host, torch_cuda

pytestmark = pytest.mark.gpu


def run_qnorm(x, gamma, eps, ldx=None):
    torch = torch_cuda()
    x = np.ascontiguousarray(x, dtype=np.float32)
    N, K = x.shape
    if ldx is not None and ldx != K:
        buf = np.zeros((N, ldx), dtype=np.float32)
        buf[:, :K] = x
        xd = to_dev(buf)
    else:
        ldx = K
        xd = to_dev(x)
    gd = None if gamma is None else to_dev(gamma)
    xq = empty_u8(qdg.q8_0_nbytes(N, K))
    qdg.qnorm_quantize_q8_0(xd, gd, eps, xq, K=K, N=N, ldx=ldx)
    torch.cuda.synchronize()
    return to_host(xq).reshape(N, -1)


@pytest.mark.parametrize("K", [32, 96, 256, 2048, 4096, 8192, 14336])
@pytest.mark.parametrize("norm", [True, False])
def test_qnorm_bit_exact(K, norm):
    N = 3
    x = synth.activations(10 + K, "qn", N, K, outlier_frac=0.01)
    gam = synth.gamma(10 + K, "qn", K) if norm else None
    got = run_qnorm(x, gam, 1e-6)
    ref = oracle.quantize_q8_0(x, gam, 1e-6)
    assert np.array_equal(got, ref)


def run_qnorm_add(x, gamma, add, eps, ldadd_pad=0):
    torch = torch_cuda()
    x = np.ascontiguousarray(x, dtype=np.float32)
    N, K = x.shape
    add = np.ascontiguousarray(add, dtype=np.float32)
    if add.ndim == 2 and ldadd_pad:
        buf = np.zeros((N, K + ldadd_pad), dtype=np.float32)
        buf[:, :K] = add
        ad, ldadd = to_dev(buf), K + ldadd_pad
    else:
        ad, ldadd = to_dev(add), (0 if add.ndim == 1 else K)
    xq = empty_u8(qdg.q8_0_nbytes(N, K))
    qdg.qnorm_add_quantize_q8_0(to_dev(x), None if gamma is None else to_dev(gamma), ad, eps, xq, K=K, N=N,
                                ldadd=ldadd)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    return to_host(xq).reshape(N, -1)


@pytest.mark.parametrize("K", [32, 256, 4096, 14336])
@pytest.mark.parametrize("norm", [True, False])
@pytest.mark.parametrize("per_row", [True, False])
def test_qnorm_add_bit_exact(K, norm, per_row):
    """RMS_NORM + MUL + ADD -> Q8_0 against the oracle, byte for byte; the
    addend is residual-like (same scale as x, 1% outliers)."""
    N = 3
    x = synth.activations(20 + K, "qa-x", N, K, outlier_frac=0.01)
    gam = synth.gamma(20 + K, "qa-g", K) if norm else None
    a = synth.activations(20 + K, "qa-a", N, K, outlier_frac=0.01)
    add = a if per_row else a[0]
    got = run_qnorm_add(x, gam, add, 1e-6, ldadd_pad=16 if per_row else 0)
    assert np.array_equal(got, oracle.quantize_q8_0(x, gam, 1e-6, add=add))


def test_qnorm_add_zero_matches_plain_entry():
    K, N = 2048, 2
    x = synth.activations(31, "qa0", N, K)
    gam = synth.gamma(31, "qa0", K)
    assert np.array_equal(run_qnorm_add(x, gam, np.zeros(K, np.float32), 1e-6), run_qnorm(x, gam, 1e-6))


def test_qnorm_many_columns_and_stride():
    K, N = 4096, 512
    x = synth.activations(4, "prefill-x", N, K)
    gam = synth.gamma(4, "prefill-g", K)
    got = run_qnorm(x, gam, 1e-5, ldx=K + 64)
    assert np.array_equal(got, oracle.quantize_q8_0(x, gam, 1e-5))


def test_qnorm_edge_values():
    K = 256
    x = np.zeros((5, K), dtype=np.float32)
    x[1] = 2.0                                        # constant vector: every q = 127
    x[2, 5] = -3.0                                    # one non-zero element
    x[3] = np.float32(1e-20)                          # tiny values, eps dominates
    x[4, ::2] = 1.0
    x[4, 1::2] = -1.0
    gam = np.ones(K, dtype=np.float32)
    for eps in (0.0, 1e-6, 1.0):
        got = run_qnorm(x[1:] if eps == 0.0 else x, gam, eps)   # eps = 0 with a zero vector is 0/0
        ref = oracle.quantize_q8_0(x[1:] if eps == 0.0 else x, gam, eps)
        assert np.array_equal(got, ref)
    # plain path on the zero vector: d = 0, q = 0
    got = run_qnorm(x, None, 0.0)
    assert np.array_equal(got, oracle.quantize_q8_0(x, None, 0.0))
    assert np.all(got[0] == 0)


def test_qnorm_subnormal_and_overflow_scales():
    K = 64
    x = np.zeros((2, K), dtype=np.float32)
    x[0, :32] = np.linspace(-1, 1, 32) * 1e-6          # d in the fp16 subnormal range
    x[1, :32] = 1e7                                    # d = 1e7/127 > 65504 -> inf scale + flag
    got = run_qnorm(x, None, 0.0)
    assert np.array_equal(got, oracle.quantize_q8_0(x, None, 0.0))
    assert qdg.qdg_device_status() == qdg.QDG_EOVERFLOW
    assert qdg.qdg_device_status() == qdg.QDG_OK      # cleared


@pytest.mark.parametrize("O,K", [(1, 32), (7, 256), (300, 4096), (64, 14336)])
def test_quantize_q4_0_bit_exact(O, K):
    torch = torch_cuda()
    w = synth.weights(O + K, "q4", O, K)
    w[0, :32] = 0.0                                   # all-zero block
    if K >= 64:
        w[0, 32:64] = 0.01                            # equal magnitudes: first one wins
        w[0, 40] = -0.01
    Wq = empty_u8(qdg.q4_0_nbytes(O, K))
    qdg.quantize_q4_0(to_dev(w), Wq)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(Wq).reshape(O, -1), oracle.quantize_q4_0(w))


def test_quantize_q4_0_leading_dimension():
    torch = torch_cuda()
    O, K, ldw = 33, 256, 320
    w = synth.weights(5, "q4-ld", O, ldw)
    Wq = empty_u8(qdg.q4_0_nbytes(O, K))
    qdg.quantize_q4_0(to_dev(w), Wq, O=O, K=K, ldw=ldw)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(Wq).reshape(O, -1), oracle.quantize_q4_0(w[:, :K]))


def test_timeout_probe_reports_and_recovers():
    torch = torch_cuda()
    qdg.qdg_debug_timeout_probe()
    assert qdg.qdg_device_status() == qdg.QDG_ETIMEOUT
    assert qdg.qdg_device_status() == qdg.QDG_OK
    # the context still works
    x = synth.activations(1, "after-timeout", 1, 256)
    assert np.array_equal(run_qnorm(x, None, 0.0), oracle.quantize_q8_0(x, None, 0.0))
