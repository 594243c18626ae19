"""GPU parity of the Q8_0-weight GEMV against the CPU oracle: exact per-block
integer sums through the test hook, fp32 outputs within
1e-5 * sum_b |d_w d_x isum_b|, grouped launches, extreme codes, PDL on/off."""
import numpy as np
import pytest

import oracle
from quantized_decode_gemv_rms_gb300 import qdg, synth
from helpers import assert_within_tol, to_dev, to_host, torch_cuda

pytestmark = pytest.mark.gpu


def problem(seed, O, K, outliers=0.0):
    w = synth.weights(seed, "W8", O, K)
    x = synth.activations(seed, "x", 1, K, outlier_frac=outliers)
    gam = synth.gamma(seed, "g", K)
    return oracle.quantize_q8_0(w, None), oracle.quantize_q8_0(x, gam, 1e-6)


def gpu_gemv_q8w(Wq, xq, O, K):
    torch = torch_cuda()
    y = torch.full((O,), float("nan"), dtype=torch.float32, device="cuda")
    qdg.q8_0_q8_0_gemv(to_dev(Wq), to_dev(xq), y, O, K)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    return to_host(y)


# one ragged segment (K = 256, 2304), whole segments (2048, 4096), 16 segments
# (K = 32768: one row slot per CTA); rows below, at and above the SM count
Q8W_SHAPES = [(1, 256), (300, 256), (37, 2304), (1000, 2048), (152, 4096), (153, 4096), (600, 6144),
              (4096, 14336), (64, 32768), (3000, 768)]


@pytest.mark.parametrize("O,K", Q8W_SHAPES)
def test_q8w_block_sums_exact(O, K):
    Wq, xq = problem(O * 5 + K, O, K)
    torch = torch_cuda()
    isum = torch.full((1, O, K // 32), -2 ** 31, dtype=torch.int32, device="cuda")
    qdg.qdg_debug_block_sums(to_dev(Wq), to_dev(xq), isum, O, K, 1, 4)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(isum), oracle.block_sums(Wq, xq, K, wtype="q8_0"))


@pytest.mark.parametrize("O,K", Q8W_SHAPES)
def test_q8w_output_within_tolerance(O, K):
    Wq, xq = problem(O * 13 + K, O, K, outliers=0.01)
    y = gpu_gemv_q8w(Wq, xq, O, K)
    _, y64, S = oracle.matvec(Wq, xq, K, threads=8, wtype="q8_0")
    assert_within_tol(y[None, :], y64, S)


def test_q8w_extreme_codes():
    """Rows of all +127, all -127 and alternating codes against activations of
    +-127: the largest block sums the format allows (32 * 127^2)."""
    K, O = 2048, 3
    nb = K // 32
    W = np.zeros((O, nb, 34), dtype=np.uint8)
    d = np.float16(0.015625).view(np.uint16)
    W[:, :, 0] = d & 0xFF
    W[:, :, 1] = d >> 8
    W[0, :, 2:] = np.int8(127).view(np.uint8)
    W[1, :, 2:] = np.int8(-127).view(np.uint8)
    W[2, :, 2:] = np.tile(np.array([127, -127], dtype=np.int8), 16).view(np.uint8)
    X = np.zeros((1, nb, 34), dtype=np.uint8)
    X[:, :, 0] = np.float16(0.5).view(np.uint16) & 0xFF
    X[:, :, 1] = np.float16(0.5).view(np.uint16) >> 8
    X[0, :, 2:] = np.tile(np.array([127, 127, -127, 127], dtype=np.int8), 8).view(np.uint8)
    W, X = W.reshape(O, -1), X.reshape(1, -1)
    y = gpu_gemv_q8w(W, X, O, K)
    _, y64, S = oracle.matvec(W, X, K, wtype="q8_0")
    assert_within_tol(y[None, :], y64, S)


def test_q8w_group_matches_single_calls():
    torch = torch_cuda()
    K = 4096
    xq = problem(6, 8, K)[1]
    xd = to_dev(xq)
    shapes = {"q": 1024, "k": 256, "v": 256}
    Wq = {n: oracle.quantize_q8_0(synth.weights(10, n, O, K), None) for n, O in shapes.items()}
    Wd = {n: to_dev(Wq[n]) for n in shapes}
    single = {}
    for n, O in shapes.items():
        y = torch.empty(O, dtype=torch.float32, device="cuda")
        qdg.q8_0_q8_0_gemv(Wd[n], xd, y, O, K)
        single[n] = y
    ys = [torch.empty(shapes[n], dtype=torch.float32, device="cuda") for n in shapes]
    qdg.q8_0_q8_0_gemv_group([Wd[n] for n in shapes], ys, list(shapes.values()), xd, K)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    for n, y in zip(shapes, ys):
        assert np.array_equal(to_host(y).view(np.uint32), to_host(single[n]).view(np.uint32)), n
        _, y64, S = oracle.matvec(Wq[n], xq, K, threads=8, wtype="q8_0")
        assert_within_tol(to_host(y)[None, :], y64, S)


def test_q8w_deterministic_and_pdl_invariant():
    torch = torch_cuda()
    O, K = 14336, 4096
    Wq, xq = problem(79, O, K)
    Wd, xd = to_dev(Wq), to_dev(xq)
    outs = []
    for pdl in (0, 1, 0):
        qdg.qdg_set_option(qdg.QDG_OPT_PDL, pdl)
        y = torch.empty(O, dtype=torch.float32, device="cuda")
        for _ in range(3):
            qdg.q8_0_q8_0_gemv(Wd, xd, y, O, K)
        torch.cuda.synchronize()
        outs.append(to_host(y))
    qdg.qdg_set_option(qdg.QDG_OPT_PDL, 0)
    assert all(np.array_equal(outs[0].view(np.uint32), o.view(np.uint32)) for o in outs[1:])
    rows = synth.sample_indices(O, "q8w-rows", O, 1024)
    _, y64, S = oracle.matvec(Wq, xq, K, rows=rows, threads=8, wtype="q8_0")
    assert_within_tol(outs[0][rows][None, :], y64, S)
