"""GPU parity of the Q4_K-weight GEMV against the CPU oracle: exact integer
sums per 32-weight sub-block through the test hook, fp32 outputs within
1e-5 * sum_b (|d_x d sc_b isum_b| + |d_x dmin m_b xsum_b|), extreme and
hand-built super-blocks, grouped launches, determinism and PDL on/off."""
import json
import os

import numpy as np
import pytest

import oracle
from quantized_decode_gemv_rms_gb300 import qdg, synth
from helpers import assert_within_tol, to_dev, to_host, torch_cuda

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_blocks.json")


def problem(seed, O, K, outliers=0.0):
    w = synth.weights(seed, "W4K", O, K)
    x = synth.activations(seed, "x", 1, K, outlier_frac=outliers)
    gam = synth.gamma(seed, "g", K)
    return oracle.quantize_q4_k(w), oracle.quantize_q8_0(x, gam, 1e-6)


def gpu_gemv_q4k(Wq, xq, O, K):
    torch = torch_cuda()
    y = torch.full((O,), float("nan"), dtype=torch.float32, device="cuda")
    qdg.q4_k_q8_0_gemv(to_dev(Wq), to_dev(xq), y, O, K)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    return to_host(y)


# one super-block (K = 256), ragged last segments (2304, 6400), whole
# segments (2048, 4096, 14336), 16 segments (K = 32768); rows below, at and
# above the SM count
Q4K_SHAPES = [(1, 256), (300, 256), (37, 2304), (1000, 2048), (152, 4096), (153, 4096), (600, 6400),
              (4096, 14336), (64, 32768), (3000, 768)]


@pytest.mark.parametrize("O,K", Q4K_SHAPES)
def test_q4k_block_sums_exact(O, K):
    Wq, xq = problem(O * 3 + K, O, K)
    torch = torch_cuda()
    isum = torch.full((1, O, K // 32), -2 ** 31, dtype=torch.int32, device="cuda")
    qdg.qdg_debug_block_sums(to_dev(Wq), to_dev(xq), isum, O, K, 1, 6)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(isum), oracle.block_sums(Wq, xq, K, wtype="q4_k"))


@pytest.mark.parametrize("O,K", Q4K_SHAPES)
def test_q4k_output_within_tolerance(O, K):
    Wq, xq = problem(O * 11 + K, O, K, outliers=0.01)
    y = gpu_gemv_q4k(Wq, xq, O, K)
    _, y64, S = oracle.matvec(Wq, xq, K, threads=8, wtype="q4_k")
    assert_within_tol(y[None, :], y64, S)


def test_q4k_hand_superblock():
    """The hand-derived super-block of the oracle's pins (every sub-block
    scale and min, including the packed high bits) against an all-ones Q8_0
    vector: y = 19248 exactly."""
    g = json.load(open(GOLDEN))["q4k_superblock"]
    blk = np.zeros(144, dtype=np.uint8)
    blk[0], blk[1] = g["d_bits"] & 0xFF, g["d_bits"] >> 8
    blk[2], blk[3] = g["dmin_bits"] & 0xFF, g["dmin_bits"] >> 8
    blk[4:16] = g["scales_bytes"]
    for j in range(8):
        for i in range(32):
            q = (i + 3 * j) % 16
            blk[16 + 32 * (j // 2) + i] |= np.uint8(q if j % 2 == 0 else q << 4)
    O, K = 5, 1024
    W = np.tile(blk, (O, K // 256))
    x = np.zeros((1, K // 32 * 34), dtype=np.uint8)
    for b in range(K // 32):
        x[0, 34 * b] = g["x_d_bits"] & 0xFF
        x[0, 34 * b + 1] = g["x_d_bits"] >> 8
        x[0, 34 * b + 2:34 * b + 34] = 1
    y = gpu_gemv_q4k(W, x, O, K)
    assert np.all(y == np.float32(g["y"] * (K // 256)))


def test_q4k_extreme_codes():
    """All codes 15 and all 0 with the largest scales and mins (63) against
    activations of +-127: the largest sub-block sums the format allows."""
    O, K = 4, 2048
    nsb = K // 256
    W = np.zeros((O, nsb, 144), dtype=np.uint8)
    d = np.float16(0.0078125).view(np.uint16)
    dm = np.float16(0.00390625).view(np.uint16)
    W[:, :, 0], W[:, :, 1] = d & 0xFF, d >> 8
    W[:, :, 2], W[:, :, 3] = dm & 0xFF, dm >> 8
    W[:, :, 4:16] = 255                       # every scale and min 63
    W[0, :, 16:] = 0xFF                        # codes 15
    W[1, :, 16:] = 0x00                        # codes 0
    W[2, :, 16:] = 0x0F                        # 15 in even sub-blocks, 0 in odd
    W[3, :, 16:] = np.tile(np.array([0xF0, 0x0F], dtype=np.uint8), 64)
    X = np.zeros((1, K // 32, 34), dtype=np.uint8)
    X[:, :, 0] = np.float16(0.5).view(np.uint16) & 0xFF
    X[:, :, 1] = np.float16(0.5).view(np.uint16) >> 8
    X[0, :, 2:] = np.tile(np.array([127, 127, -127, 127], dtype=np.int8), 8).view(np.uint8)
    W, X = W.reshape(O, -1), X.reshape(1, -1)
    y = gpu_gemv_q4k(W, X, O, K)
    _, y64, S = oracle.matvec(W, X, K, wtype="q4_k")
    assert_within_tol(y[None, :], y64, S)


def test_q4k_group_matches_single_calls():
    torch = torch_cuda()
    K = 4096
    xq = problem(6, 8, K)[1]
    xd = to_dev(xq)
    shapes = {"q": 1024, "k": 256, "v": 256}
    Wq = {n: oracle.quantize_q4_k(synth.weights(12, n, O, K)) for n, O in shapes.items()}
    Wd = {n: to_dev(Wq[n]) for n in shapes}
    single = {}
    for n, O in shapes.items():
        y = torch.empty(O, dtype=torch.float32, device="cuda")
        qdg.q4_k_q8_0_gemv(Wd[n], xd, y, O, K)
        single[n] = y
    ys = [torch.empty(shapes[n], dtype=torch.float32, device="cuda") for n in shapes]
    qdg.q4_k_q8_0_gemv_group([Wd[n] for n in shapes], ys, list(shapes.values()), xd, K)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    for n, y in zip(shapes, ys):
        assert np.array_equal(to_host(y).view(np.uint32), to_host(single[n]).view(np.uint32)), n
        _, y64, S = oracle.matvec(Wq[n], xq, K, threads=8, wtype="q4_k")
        assert_within_tol(to_host(y)[None, :], y64, S)


def test_q4k_deterministic_and_pdl_invariant():
    torch = torch_cuda()
    O, K = 14336, 4096
    Wq, xq = problem(81, O, K)
    Wd, xd = to_dev(Wq), to_dev(xq)
    outs = []
    for pdl in (0, 1, 0):
        qdg.qdg_set_option(qdg.QDG_OPT_PDL, pdl)
        y = torch.empty(O, dtype=torch.float32, device="cuda")
        for _ in range(3):
            qdg.q4_k_q8_0_gemv(Wd, xd, y, O, K)
        torch.cuda.synchronize()
        outs.append(to_host(y))
    qdg.qdg_set_option(qdg.QDG_OPT_PDL, 0)
    assert all(np.array_equal(outs[0].view(np.uint32), o.view(np.uint32)) for o in outs[1:])
    rows = synth.sample_indices(O, "q4k-rows", O, 1024)
    _, y64, S = oracle.matvec(Wq, xq, K, rows=rows, threads=8, wtype="q4_k")
    assert_within_tol(outs[0][rows][None, :], y64, S)


@pytest.mark.parametrize("O,K", [(1, 256), (77, 2304), (512, 4096), (3, 14336)])
def test_quantize_q4_k_matches_oracle_bytes(O, K):
    """The load-time quantizer on the GPU, byte for byte against the oracle's
    (same reading, every step one IEEE fp32 operation); includes zero,
    constant and all-negative super-blocks."""
    torch = torch_cuda()
    w = synth.weights(O + K, "q4k-quant", O, K)
    w[0, :256] = 0.0
    if O > 2:
        w[1, 256 % K:256 % K + 256] = 0.75
        w[2, :256] = -np.abs(w[2, :256]) - 0.01
    Wq = torch.zeros(O * (K // 256) * 144, dtype=torch.uint8, device="cuda")
    qdg.quantize_q4_k(to_dev(w), Wq, O=O, K=K)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(Wq).reshape(O, -1), oracle.quantize_q4_k(w))


@pytest.mark.parametrize("wtype", ["q4_k", "q5_k"])
def test_kquant_rows_in_two_chunks(wtype):
    """More rows per CTA than one chunk of partial sums holds (K = 32768:
    16 segments, 192 rows a chunk; O = 29500 gives 194-195 rows a CTA), so
    each CTA refills its ring across a chunk boundary.  Super-blocks are
    seeded random bytes with fixed finite scales (every code, scale and min
    byte pattern is a valid block); exact block sums and outputs on sampled
    rows against the oracle."""
    torch = torch_cuda()
    O, K = 29500, 32768
    sbb = 144 if wtype == "q4_k" else 176
    nsb = K // 256
    W = synth.raw_bytes(29, f"{wtype}-chunks", O * nsb * sbb).reshape(O, nsb, sbb)
    W[:, :, 0:2] = np.frombuffer(np.float16(0.003).tobytes(), dtype=np.uint8)
    W[:, :, 2:4] = np.frombuffer(np.float16(0.001).tobytes(), dtype=np.uint8)
    W = W.reshape(O, -1)
    xq = oracle.quantize_q8_0(synth.activations(29, "xc", 1, K), None)
    Wd, xd = to_dev(W), to_dev(xq)
    rows = synth.sample_indices(29, "rows-chunks", O, 384)
    path = 6 if wtype == "q4_k" else 7
    isum = torch.full((1, O, K // 32), -2 ** 31, dtype=torch.int32, device="cuda")
    qdg.qdg_debug_block_sums(Wd, xd, isum, O, K, 1, path)
    y = torch.full((O,), float("nan"), dtype=torch.float32, device="cuda")
    gemv = qdg.q4_k_q8_0_gemv if wtype == "q4_k" else qdg.q5_k_q8_0_gemv
    gemv(Wd, xd, y, O, K)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    assert np.array_equal(to_host(isum)[:, rows], oracle.block_sums(W[rows], xq, K, wtype=wtype))
    _, y64, S = oracle.matvec(W, xq, K, rows=rows, threads=8, wtype=wtype)
    assert_within_tol(to_host(y)[rows][None, :], y64, S)
