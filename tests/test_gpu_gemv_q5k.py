"""GPU parity of the Q5_K-weight GEMV and its load-time quantizer against the
CPU oracle: exact integer sums per 32-weight sub-block through the test hook,
fp32 outputs within 1e-5 * sum_b (|d_x d sc_b isum_b| + |d_x dmin m_b
xsum_b|), the hand-derived super-block, the largest codes the format holds,
grouped launches, determinism with and without PDL, and the quantizer's bytes."""
import json
import os

import numpy as np
import pytest

import oracle
from quantized_decode_gemv_rms_gb300 import qdg, synth
from helpers import assert_within_tol, to_dev, to_host, torch_cuda

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_blocks.json")
SB = 176        # bytes of a Q5_K super-block


def problem(seed, O, K, outliers=0.0):
    w = synth.weights(seed, "W5K", O, K)
    x = synth.activations(seed, "x5", 1, K, outlier_frac=outliers)
    gam = synth.gamma(seed, "g5", K)
    return oracle.quantize_q5_k(w), oracle.quantize_q8_0(x, gam, 1e-6)


def gpu_gemv_q5k(Wq, xq, O, K):
    torch = torch_cuda()
    y = torch.full((O,), float("nan"), dtype=torch.float32, device="cuda")
    qdg.q5_k_q8_0_gemv(to_dev(Wq), to_dev(xq), y, O, K)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    return to_host(y)


# one super-block (K = 256), ragged last segments (2304, 6400: 1 and 1 of 8
# super-blocks), whole segments (2048, 4096, 14336), 16 segments (32768);
# rows below, at and above the SM count
Q5K_SHAPES = [(1, 256), (300, 256), (37, 2304), (1000, 2048), (152, 4096), (153, 4096), (600, 6400),
              (4096, 14336), (64, 32768), (3000, 768)]


@pytest.mark.parametrize("O,K", Q5K_SHAPES)
def test_q5k_block_sums_exact(O, K):
    Wq, xq = problem(O * 5 + K, O, K)
    torch = torch_cuda()
    isum = torch.full((1, O, K // 32), -2 ** 31, dtype=torch.int32, device="cuda")
    qdg.qdg_debug_block_sums(to_dev(Wq), to_dev(xq), isum, O, K, 1, 7)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(isum), oracle.block_sums(Wq, xq, K, wtype="q5_k"))


@pytest.mark.parametrize("O,K", Q5K_SHAPES)
def test_q5k_output_within_tolerance(O, K):
    Wq, xq = problem(O * 13 + K, O, K, outliers=0.01)
    y = gpu_gemv_q5k(Wq, xq, O, K)
    _, y64, S = oracle.matvec(Wq, xq, K, threads=8, wtype="q5_k")
    assert_within_tol(y[None, :], y64, S)


def test_q5k_hand_superblock():
    """The hand-derived super-block of the oracle's pins (codes 0..31 in every
    sub-block, top bits in qh) against an all-ones Q8_0 vector: y = 41392 a
    super-block, exactly."""
    g = json.load(open(GOLDEN))["q5k_superblock"]
    blk = np.zeros(SB, dtype=np.uint8)
    blk[0], blk[1] = g["d_bits"] & 0xFF, g["d_bits"] >> 8
    blk[2], blk[3] = g["dmin_bits"] & 0xFF, g["dmin_bits"] >> 8
    blk[4:16] = g["scales_bytes"]
    for j in range(8):
        for i in range(32):
            q = (i + 3 * j) % 32
            blk[48 + 32 * (j // 2) + i] |= np.uint8((q & 15) if j % 2 == 0 else (q & 15) << 4)
            blk[16 + i] |= np.uint8((q >> 4) << j)
    for k, v in g["spot_bytes"].items():
        assert int(blk[int(k)]) == v
    O, K = 5, 1024
    W = np.tile(blk, (O, K // 256))
    x = np.zeros((1, K // 32 * 34), dtype=np.uint8)
    for b in range(K // 32):
        x[0, 34 * b] = g["x_d_bits"] & 0xFF
        x[0, 34 * b + 1] = g["x_d_bits"] >> 8
        x[0, 34 * b + 2:34 * b + 34] = 1
    y = gpu_gemv_q5k(W, x, O, K)
    assert np.all(y == np.float32(g["y"] * (K // 256)))


def test_q5k_extreme_codes():
    """Codes 31 and 0 (every qh bit set or clear, nibbles 15 or 0) with the
    largest scales and mins (63) against activations of +-127: the largest
    sub-block sums the format allows, and rows whose top bits differ between
    the two sub-blocks a lane reads."""
    O, K = 5, 2048
    nsb = K // 256
    W = np.zeros((O, nsb, SB), dtype=np.uint8)
    d = np.float16(0.0078125).view(np.uint16)
    dm = np.float16(0.00390625).view(np.uint16)
    W[:, :, 0], W[:, :, 1] = d & 0xFF, d >> 8
    W[:, :, 2], W[:, :, 3] = dm & 0xFF, dm >> 8
    W[:, :, 4:16] = 255                        # every scale and min 63
    W[0, :, 16:] = 0xFF                        # codes 31
    W[1, :, 16:] = 0x00                        # codes 0
    W[2, :, 16:48] = 0x55                      # top bit in even sub-blocks only
    W[2, :, 48:] = 0xFF                        # -> 31 in even sub-blocks, 15 in odd
    W[3, :, 16:48] = 0xAA                      # top bit in odd sub-blocks only
    W[3, :, 48:] = 0x0F                        # -> 15 in even, 16 in odd
    W[4, :, 16:48] = np.tile(np.array([0x0F, 0xF0], dtype=np.uint8), 16)
    W[4, :, 48:] = np.tile(np.array([0xF0, 0x0F], dtype=np.uint8), 64)
    X = np.zeros((1, K // 32, 34), dtype=np.uint8)
    X[:, :, 0] = np.float16(0.5).view(np.uint16) & 0xFF
    X[:, :, 1] = np.float16(0.5).view(np.uint16) >> 8
    X[0, :, 2:] = np.tile(np.array([127, 127, -127, 127], dtype=np.int8), 8).view(np.uint8)
    W, X = W.reshape(O, -1), X.reshape(1, -1)
    torch = torch_cuda()
    isum = torch.full((1, O, K // 32), -2 ** 31, dtype=torch.int32, device="cuda")
    qdg.qdg_debug_block_sums(to_dev(W), to_dev(X), isum, O, K, 1, 7)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(isum), oracle.block_sums(W, X, K, wtype="q5_k"))
    y = gpu_gemv_q5k(W, X, O, K)
    _, y64, S = oracle.matvec(W, X, K, wtype="q5_k")
    assert_within_tol(y[None, :], y64, S)


def test_q5k_group_matches_single_calls():
    torch = torch_cuda()
    K = 4096
    xq = problem(7, 8, K)[1]
    xd = to_dev(xq)
    shapes = {"q": 1024, "k": 256, "v": 256}
    Wq = {n: oracle.quantize_q5_k(synth.weights(13, n, O, K)) for n, O in shapes.items()}
    Wd = {n: to_dev(Wq[n]) for n in shapes}
    single = {}
    for n, O in shapes.items():
        y = torch.empty(O, dtype=torch.float32, device="cuda")
        qdg.q5_k_q8_0_gemv(Wd[n], xd, y, O, K)
        single[n] = y
    ys = [torch.empty(shapes[n], dtype=torch.float32, device="cuda") for n in shapes]
    qdg.q5_k_q8_0_gemv_group([Wd[n] for n in shapes], ys, list(shapes.values()), xd, K)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    for n, y in zip(shapes, ys):
        assert np.array_equal(to_host(y).view(np.uint32), to_host(single[n]).view(np.uint32)), n
        _, y64, S = oracle.matvec(Wq[n], xq, K, threads=8, wtype="q5_k")
        assert_within_tol(to_host(y)[None, :], y64, S)


def test_q5k_deterministic_and_pdl_invariant():
    torch = torch_cuda()
    O, K = 14336, 4096
    Wq, xq = problem(82, O, K)
    Wd, xd = to_dev(Wq), to_dev(xq)
    outs = []
    for pdl in (0, 1, 0):
        qdg.qdg_set_option(qdg.QDG_OPT_PDL, pdl)
        y = torch.empty(O, dtype=torch.float32, device="cuda")
        for _ in range(3):
            qdg.q5_k_q8_0_gemv(Wd, xd, y, O, K)
        torch.cuda.synchronize()
        outs.append(to_host(y))
    qdg.qdg_set_option(qdg.QDG_OPT_PDL, 0)
    assert all(np.array_equal(outs[0].view(np.uint32), o.view(np.uint32)) for o in outs[1:])
    rows = synth.sample_indices(O, "q5k-rows", O, 1024)
    _, y64, S = oracle.matvec(Wq, xq, K, rows=rows, threads=8, wtype="q5_k")
    assert_within_tol(outs[0][rows][None, :], y64, S)


@pytest.mark.parametrize("O,K", [(1, 256), (77, 2304), (512, 4096), (3, 14336)])
def test_quantize_q5_k_matches_oracle_bytes(O, K):
    """The load-time quantizer on the GPU, byte for byte against the oracle's
    (same reading, every step one IEEE fp32 operation); includes zero,
    constant and all-negative super-blocks."""
    torch = torch_cuda()
    w = synth.weights(O + K, "q5k-quant", O, K)
    w[0, :256] = 0.0
    if O > 2:
        w[1, 256 % K:256 % K + 256] = 0.75
        w[2, :256] = -np.abs(w[2, :256]) - 0.01
    Wq = torch.zeros(O * (K // 256) * SB, dtype=torch.uint8, device="cuda")
    qdg.quantize_q5_k(to_dev(w), Wq, O=O, K=K)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(Wq).reshape(O, -1), oracle.quantize_q5_k(w))
