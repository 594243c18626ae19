"""GPU parity of the product kernels (batch-1 GEMV and small-N) against the
CPU oracle: exact per-block integer sums through the test hook, fp32 outputs
within 1e-5 * sum_b |d_w d_x isum_b|, determinism, PDL on/off."""
import numpy as np
import pytest

import oracle
from quantized_decode_gemv_rms_gb300 import qdg, synth
from helpers import assert_within_tol, empty_u8, to_dev, to_host, torch_cuda

pytestmark = pytest.mark.gpu


def problem(seed, O, K, N, norm=True, outliers=0.0):
    w = synth.weights(seed, "W", O, K)
    x = synth.activations(seed, "x", N, K, outlier_frac=outliers)
    gam = synth.gamma(seed, "g", K) if norm else None
    Wq = oracle.quantize_q4_0(w)
    xq = oracle.quantize_q8_0(x, gam, 1e-6)
    return Wq, xq


def gpu_gemv(Wq, xq, O, K):
    torch = torch_cuda()
    y = torch.empty(O, dtype=torch.float32, device="cuda")
    qdg.q4_0_q8_0_gemv(to_dev(Wq), to_dev(xq), y, O, K)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    return to_host(y)


def gpu_small_n(Wq, xq, O, K, N, ldy=None):
    torch = torch_cuda()
    ldy = O if ldy is None else ldy
    y = torch.full((N, ldy), float("nan"), dtype=torch.float32, device="cuda")
    qdg.q4_0_q8_0_gemm_small_n(to_dev(Wq), to_dev(xq), y, ldy, O, K, N)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    out = to_host(y)
    if ldy > O:
        assert np.all(np.isnan(out[:, O:])), "wrote past O inside the leading dimension"
    return out[:, :O]


def gpu_block_sums(Wq, xq, O, K, N, path):
    torch = torch_cuda()
    isum = torch.full((N, O, K // 32), -2 ** 31, dtype=torch.int32, device="cuda")
    qdg.qdg_debug_block_sums(to_dev(Wq), to_dev(xq), isum, O, K, N, path)
    torch.cuda.synchronize()
    return to_host(isum)


GEMV_SHAPES = [(256, 256), (1, 256), (37, 512), (1000, 2048), (152, 4096), (1024, 4096), (153, 4096),
               (600, 6144), (4096, 14336), (64, 32768), (3000, 768)]


@pytest.mark.parametrize("O,K", GEMV_SHAPES)
def test_gemv_block_sums_exact(O, K):
    Wq, xq = problem(O * 7 + K, O, K, 1)
    got = gpu_block_sums(Wq, xq, O, K, 1, 0)
    assert np.array_equal(got, oracle.block_sums(Wq, xq, K))


@pytest.mark.parametrize("O,K", GEMV_SHAPES)
def test_gemv_output_within_tolerance(O, K):
    Wq, xq = problem(O * 11 + K, O, K, 1, outliers=0.01)
    y = gpu_gemv(Wq, xq, O, K)
    _, y64, S = oracle.matvec(Wq, xq, K, threads=8)
    assert_within_tol(y[None, :], y64, S)


def test_gemv_deterministic_and_pdl_invariant():
    torch = torch_cuda()
    O, K = 4096, 4096
    Wq, xq = problem(77, O, K, 1)
    Wd, xd = to_dev(Wq), to_dev(xq)
    outs = []
    for pdl in (0, 1, 0):
        qdg.qdg_set_option(qdg.QDG_OPT_PDL, pdl)
        y = torch.empty(O, dtype=torch.float32, device="cuda")
        for _ in range(3):
            qdg.q4_0_q8_0_gemv(Wd, xd, y, O, K)
        torch.cuda.synchronize()
        outs.append(to_host(y))
    qdg.qdg_set_option(qdg.QDG_OPT_PDL, 0)
    assert all(np.array_equal(outs[0].view(np.uint32), o.view(np.uint32)) for o in outs[1:])


def test_gemv_special_blocks():
    """All-zero codes -> -8 d_w sum(q_x); all-8 -> 0; all-15 -> 7 d_w sum(q_x)."""
    K = 512
    O = 3
    rng = np.random.default_rng(1)
    xq = oracle.quantize_q8_0(rng.standard_normal((1, K)).astype(np.float32), None)
    W = np.zeros((O, K // 32 * 18), dtype=np.uint8)
    d = np.array([np.float16(0.25).view(np.uint16)], dtype=np.uint16).view(np.uint8)
    for r, byte in enumerate((0x00, 0x88, 0xFF)):
        for b in range(K // 32):
            W[r, b * 18:b * 18 + 2] = d
            W[r, b * 18 + 2:b * 18 + 18] = byte
    y = gpu_gemv(W, xq, O, K)
    _, y64, S = oracle.matvec(W, xq, K)
    assert_within_tol(y[None, :], y64, S)
    assert y[1] == 0.0


# Covers one CTA per row range with 16 row slots (K = 256), 2 slots (K = 2048),
# one slot (K = 4096), and clusters of 2 (K = 4352 split 8 + 9 chunks, 6144,
# 8192), 4 (K = 14336) and 8 CTAs (K = 32768); ragged row tiles throughout.
SMALLN_SHAPES = [(256, 256), (2500, 256), (33, 512), (100, 4096), (1000, 2048), (17, 4352), (300, 6144),
                 (1, 8192), (4096, 14336), (14336, 4096), (40, 32768)]


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("O,K", SMALLN_SHAPES)
def test_small_n_block_sums_exact(O, K, N):
    if O * K * N > 14336 * 4096 * 2 and N not in (2, 8):
        pytest.skip("large shapes: N in {2, 8} suffice")
    Wq, xq = problem(O + K + N, O, K, N)
    got = gpu_block_sums(Wq, xq, O, K, N, 1)
    assert np.array_equal(got, oracle.block_sums(Wq, xq, K))


@pytest.mark.parametrize("N", [1, 2, 4, 7, 8])
@pytest.mark.parametrize("O,K", SMALLN_SHAPES)
def test_small_n_output_within_tolerance(O, K, N):
    Wq, xq = problem(O * 3 + K + N, O, K, N, outliers=0.01)
    rows = None if O <= 4096 else synth.sample_indices(O, "rows", O, 2048)
    y = gpu_small_n(Wq, xq, O, K, N, ldy=O + 5)
    _, y64, S = oracle.matvec(Wq, xq, K, rows=rows, threads=8)
    assert_within_tol(y if rows is None else y[:, rows], y64, S)


def _q8_blocks(codes, d):
    """Q8_0 rows from int8 codes [N][K] and one fp16 scale per row."""
    N, K = codes.shape
    out = np.zeros((N, K // 32, 34), dtype=np.uint8)
    out[:, :, 0:2] = np.array([np.float16(v) for v in d], dtype=np.float16).view(np.uint8).reshape(N, 1, 2)
    out[:, :, 2:] = codes.reshape(N, K // 32, 32).astype(np.int8).view(np.uint8)
    return out.reshape(N, -1)


@pytest.mark.parametrize("K", [4096, 8192])
def test_small_n_extreme_codes(K):
    """Largest block sums the formats allow (|q_x| = 127 against nibbles 0
    and 15), mixed with zero blocks and random ones, in every column."""
    O, N = 48, 8
    rng = np.random.default_rng(K)
    W = np.zeros((O, K // 32, 18), dtype=np.uint8)
    W[:, :, 0:2] = np.array([0.125], dtype=np.float16).view(np.uint8)
    patterns = [0x00, 0xFF, 0x88, 0x0F, 0xF0, None]
    for r in range(O):
        p = patterns[r % len(patterns)]
        W[r, :, 2:] = rng.integers(0, 256, (K // 32, 16)) if p is None else p
    W = W.reshape(O, -1)
    codes = np.empty((N, K), dtype=np.int64)
    codes[0], codes[1] = 127, -127
    codes[2] = np.where(np.arange(K) % 2 == 0, 127, -127)
    codes[3] = 0
    codes[4:] = rng.integers(-127, 128, (N - 4, K))
    xq = _q8_blocks(codes, [0.5, 0.25, 1.0, 2.0, 0.03125, 1.5, 0.75, 3.0])
    got = gpu_block_sums(W, xq, O, K, N, 1)
    assert np.array_equal(got, oracle.block_sums(W, xq, K))
    y = gpu_small_n(W, xq, O, K, N)
    _, y64, S = oracle.matvec(W, xq, K)
    assert_within_tol(y, y64, S)


def test_small_n_one_column_matches_gemv_tolerance():
    O, K = 2048, 4096
    Wq, xq = problem(5, O, K, 1)
    a = gpu_gemv(Wq, xq, O, K)
    b = gpu_small_n(Wq, xq, O, K, 1)[0]
    _, y64, S = oracle.matvec(Wq, xq, K, threads=8)
    assert_within_tol(a[None], y64, S)
    assert_within_tol(b[None], y64, S)


FUSED_SHAPES = [(256, 256), (37, 512), (1000, 2048), (4096, 4096), (153, 6144), (4096, 14336), (64, 16384)]


@pytest.mark.parametrize("norm", [True, False])
@pytest.mark.parametrize("O,K", FUSED_SHAPES)
def test_fused_norm_gemv(O, K, norm):
    """Fused RMSNorm*gamma -> Q8_0 -> GEMV: activations bit-identical to the
    standalone quantizer and to the oracle, y bit-identical to the unfused GEMV
    on those activations, and within tolerance of the oracle."""
    torch = torch_cuda()
    seed = O + K + int(norm)
    w = synth.weights(seed, "W", O, K)
    x = synth.activations(seed, "x", 1, K, outlier_frac=0.01)
    gam = synth.gamma(seed, "g", K) if norm else None
    Wd = empty_u8(qdg.q4_0_nbytes(O, K))
    qdg.quantize_q4_0(to_dev(w), Wd)
    xd = to_dev(x[0])
    gd = None if gam is None else to_dev(gam)
    xq_sep = empty_u8(qdg.q8_0_nbytes(1, K))
    qdg.qnorm_quantize_q8_0(xd, gd, 1e-6, xq_sep)
    y_sep = torch.empty(O, dtype=torch.float32, device="cuda")
    qdg.q4_0_q8_0_gemv(Wd, xq_sep, y_sep, O, K)
    xq_fused = torch.zeros(qdg.q8_0_nbytes(1, K), dtype=torch.uint8, device="cuda")
    y_fused = torch.empty(O, dtype=torch.float32, device="cuda")
    before = qdg.qdg_launch_count(5)
    qdg.q4_0_gemv_rmsnorm(Wd, xd, gd, 1e-6, y_fused, O, K, xq_out=xq_fused)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    assert qdg.qdg_launch_count(5) == before + 1
    xq_ref = oracle.quantize_q8_0(x, gam, 1e-6)
    assert np.array_equal(to_host(xq_fused).reshape(1, -1), xq_ref)
    assert np.array_equal(to_host(xq_sep).reshape(1, -1), xq_ref)
    a, b = to_host(y_fused), to_host(y_sep)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    Wq_ref = oracle.quantize_q4_0(w)
    assert np.array_equal(to_host(Wd).reshape(O, -1), Wq_ref)
    _, y64, S = oracle.matvec(Wq_ref, xq_ref, K, threads=8)
    assert_within_tol(a[None], y64, S)


def test_fused_without_xq_out_and_with_pdl():
    torch = torch_cuda()
    O, K = 2048, 4096
    w = synth.weights(3, "W", O, K)
    x = synth.activations(3, "x", 1, K)
    gam = synth.gamma(3, "g", K)
    Wd = empty_u8(qdg.q4_0_nbytes(O, K))
    qdg.quantize_q4_0(to_dev(w), Wd)
    torch.cuda.synchronize()
    outs = []
    for pdl in (0, 1):
        qdg.qdg_set_option(qdg.QDG_OPT_PDL, pdl)
        y = torch.empty(O, dtype=torch.float32, device="cuda")
        for _ in range(3):
            qdg.q4_0_gemv_rmsnorm(Wd, to_dev(x[0]), to_dev(gam), 1e-6, y, O, K)
        torch.cuda.synchronize()
        outs.append(to_host(y))
    qdg.qdg_set_option(qdg.QDG_OPT_PDL, 0)
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    xq_ref = oracle.quantize_q8_0(x, gam, 1e-6)
    _, y64, S = oracle.matvec(oracle.quantize_q4_0(w), xq_ref, K, threads=8)
    assert_within_tol(outs[0][None], y64, S)


@pytest.mark.parametrize("Os,K", [((4096, 1024, 1024), 4096), ((14336, 14336), 4096), ((37, 1, 300, 5), 2048),
                                  ((64, 128), 14336)])
def test_fused_group_matches_single(Os, K):
    """One grouped launch over matrices sharing the input equals one fused
    launch per matrix, bit for bit, and matches the oracle."""
    torch = torch_cuda()
    seed = sum(Os) + K
    x = synth.activations(seed, "x", 1, K, outlier_frac=0.01)
    gam = synth.gamma(seed, "g", K)
    xd, gd = to_dev(x[0]), to_dev(gam)
    Ws, ws = [], []
    for i, O in enumerate(Os):
        w = synth.weights(seed, f"W{i}", O, K)
        Wd = empty_u8(qdg.q4_0_nbytes(O, K))
        qdg.quantize_q4_0(to_dev(w), Wd)
        Ws.append(Wd)
        ws.append(w)
    ys_group = [torch.empty(O, dtype=torch.float32, device="cuda") for O in Os]
    xq = torch.zeros(qdg.q8_0_nbytes(1, K), dtype=torch.uint8, device="cuda")
    qdg.q4_0_gemv_rmsnorm_group(Ws, ys_group, Os, xd, gd, 1e-6, K, xq_out=xq)
    ys_single = []
    for Wd, O in zip(Ws, Os):
        y = torch.empty(O, dtype=torch.float32, device="cuda")
        qdg.q4_0_gemv_rmsnorm(Wd, xd, gd, 1e-6, y, O, K)
        ys_single.append(y)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    xq_ref = oracle.quantize_q8_0(x, gam, 1e-6)
    assert np.array_equal(to_host(xq).reshape(1, -1), xq_ref)
    for i, (a, b) in enumerate(zip(ys_group, ys_single)):
        ga, sb = to_host(a), to_host(b)
        assert np.array_equal(ga.view(np.uint32), sb.view(np.uint32)), f"matrix {i}"
        rows = None if Os[i] <= 2048 else synth.sample_indices(seed, f"r{i}", Os[i], 1024)
        Wq_ref = oracle.quantize_q4_0(ws[i] if rows is None else ws[i][rows])
        _, y64, S = oracle.matvec(Wq_ref, xq_ref, K, threads=8)
        assert_within_tol((ga if rows is None else ga[rows])[None], y64, S)


@pytest.mark.parametrize("Os,K", [((4096, 1024, 1024), 4096), ((37, 1, 300, 5), 2048), ((64, 128), 14336),
                                  ((100, 50), 32768)])
def test_gemv_group_matches_single(Os, K):
    """One grouped GEMV launch over matrices sharing a Q8_0 vector equals one
    launch per matrix, bit for bit, and matches the oracle."""
    torch = torch_cuda()
    seed = 7 * sum(Os) + K
    x = synth.activations(seed, "x", 1, K)
    xq_ref = oracle.quantize_q8_0(x, synth.gamma(seed, "g", K), 1e-6)
    xd = to_dev(xq_ref)
    Wqs = [oracle.quantize_q4_0(synth.weights(seed, f"W{i}", O, K)) for i, O in enumerate(Os)]
    Wds = [to_dev(w) for w in Wqs]
    ys = [torch.empty(O, dtype=torch.float32, device="cuda") for O in Os]
    qdg.q4_0_q8_0_gemv_group(Wds, ys, Os, xd, K)
    singles = []
    for Wd, O in zip(Wds, Os):
        y = torch.empty(O, dtype=torch.float32, device="cuda")
        qdg.q4_0_q8_0_gemv(Wd, xd, y, O, K)
        singles.append(y)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    for i, (a, b) in enumerate(zip(ys, singles)):
        ga, sb = to_host(a), to_host(b)
        assert np.array_equal(ga.view(np.uint32), sb.view(np.uint32)), f"matrix {i}"
        _, y64, S = oracle.matvec(Wqs[i], xq_ref, K, threads=8)
        assert_within_tol(ga[None], y64, S)


def raw_blocks(seed, name, O, K, block_bytes, d):
    """Seeded random rows of 32-element blocks (Q4_0: 18 bytes, Q8_0: 34)
    with a fixed finite fp16 scale in every block; Q8_0 codes of -128, which
    the quantizer never writes, become -127."""
    W = synth.raw_bytes(seed, name, O * (K // 32) * block_bytes).reshape(O, K // 32, block_bytes)
    W[:, :, 0:2] = np.frombuffer(np.float16(d).tobytes(), dtype=np.uint8)
    if block_bytes == 34:
        codes = W[:, :, 2:]
        codes[codes == 0x80] = 0x81
    return W.reshape(O, -1)


@pytest.mark.parametrize("kind", ["gemv", "fused", "q8w"])
def test_rows_in_two_chunks(kind):
    """More rows per CTA than one chunk of partial sums holds, so each CTA
    fills its ring again at the chunk boundary: the Q4_0 GEMV at K = 32768
    (256 rows a chunk; O = 39500 gives 259-260 rows a CTA), its fused form at
    K = 16384 (512 rows; O = 78000: 513-514) and the Q8_0-weight GEMV at
    K = 32768 (128 rows; O = 19800: 130-131).  Exact block sums of the
    product kernel and outputs on sampled rows against the oracle."""
    torch = torch_cuda()
    O, K = {"gemv": (39500, 32768), "fused": (78000, 16384), "q8w": (19800, 32768)}[kind]
    q8w = kind == "q8w"
    W = raw_blocks(O, "Wc", O, K, 34 if q8w else 18, 0.0005 if q8w else 0.004)
    x = synth.activations(O, "xc", 1, K, outlier_frac=0.01)
    gam = synth.gamma(O, "gc", K)
    xq = oracle.quantize_q8_0(x, gam, 1e-6)
    Wd, xd = to_dev(W), to_dev(xq)
    rows = synth.sample_indices(O, "rows-c", O, 384)
    isum = torch.full((1, O, K // 32), -2 ** 31, dtype=torch.int32, device="cuda")
    qdg.qdg_debug_block_sums(Wd, xd, isum, O, K, 1, 4 if q8w else 0)
    y = torch.full((O,), float("nan"), dtype=torch.float32, device="cuda")
    if kind == "gemv":
        qdg.q4_0_q8_0_gemv(Wd, xd, y, O, K)
    elif kind == "q8w":
        qdg.q8_0_q8_0_gemv(Wd, xd, y, O, K)
    else:
        qdg.q4_0_gemv_rmsnorm(Wd, to_dev(x[0]), to_dev(gam), 1e-6, y, O, K)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    wtype = "q8_0" if q8w else "q4_0"
    assert np.array_equal(to_host(isum)[:, rows], oracle.block_sums(W[rows], xq, K, wtype=wtype))
    _, y64, S = oracle.matvec(W, xq, K, rows=rows, threads=8, wtype=wtype)
    assert_within_tol(to_host(y)[rows][None, :], y64, S)


@pytest.mark.parametrize("layout,O,K", [("plain", 20000, 4096), ("plain", 5000, 14336), ("seg", 15000, 4096)])
@pytest.mark.parametrize("N", [3, 8])
def test_small_n_rows_in_two_batches(layout, O, K, N):
    """More row tiles per CTA (or cluster) than one batch of partial sums
    holds, so the partials are combined twice: plain layout, 8 tiles a batch
    (K = 4096, one CTA: 131-132 rows; K = 14336, clusters of four CTAs:
    131-132 rows a cluster, the cluster form's double-buffered batch
    partials); segment layout, 6 tiles a batch (K = 4096: 98-99 rows).  Exact
    block sums and outputs on sampled rows."""
    torch = torch_cuda()
    Wq = raw_blocks(O + K + N, "Wb", O, K, 18, 0.004)
    xq = oracle.quantize_q8_0(synth.activations(O + N, "xb", N, K, outlier_frac=0.01), None)
    seg = layout == "seg"
    Wd, xd = to_dev(oracle.repack_q4_0_seg(Wq, K) if seg else Wq), to_dev(xq)
    isum = torch.full((N, O, K // 32), -2 ** 31, dtype=torch.int32, device="cuda")
    qdg.qdg_debug_block_sums(Wd, xd, isum, O, K, N, 5 if seg else 1)
    y = torch.full((N, O), float("nan"), dtype=torch.float32, device="cuda")
    if seg:
        qdg.q4_0s_q8_0_gemm_small_n(Wd, xd, y, O, O, K, N)
    else:
        qdg.q4_0_q8_0_gemm_small_n(Wd, xd, y, O, O, K, N)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    rows = synth.sample_indices(O + N, "rows-b", O, 512)
    assert np.array_equal(to_host(isum)[:, rows], oracle.block_sums(Wq[rows], xq, K))
    _, y64, S = oracle.matvec(Wq, xq, K, rows=rows, threads=8)
    assert_within_tol(to_host(y)[:, rows], y64, S)
