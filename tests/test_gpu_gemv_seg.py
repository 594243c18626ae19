"""GPU parity of the segment layout (load-time repack of Q4_0 rows) and of the
GEMV that reads it: the repack byte for byte against the oracle's, exact
per-block integer sums, fp32 outputs within 1e-5 * sum_b |d_w d_x isum_b|,
grouped and concatenated matrices, PDL on/off."""
import numpy as np
import pytest

import oracle
from quantized_decode_gemv_rms_gb300 import qdg, synth
from helpers import assert_within_tol, empty_u8, to_dev, to_host, torch_cuda

pytestmark = pytest.mark.gpu


def problem(seed, O, K, outliers=0.0):
    w = synth.weights(seed, "W", O, K)
    x = synth.activations(seed, "x", 1, K, outlier_frac=outliers)
    gam = synth.gamma(seed, "g", K)
    return oracle.quantize_q4_0(w), oracle.quantize_q8_0(x, gam, 1e-6)


def gpu_repack(Wq, O, K):
    torch = torch_cuda()
    Wr = empty_u8(qdg.q4_0_seg_nbytes(O, K))
    Wr.fill_(0xA5)
    qdg.q4_0_repack_seg(to_dev(Wq), Wr, O, K)
    torch.cuda.synchronize()
    return to_host(Wr).reshape(O, -1)


def gpu_gemv_seg(Wr, xq, O, K):
    torch = torch_cuda()
    y = torch.full((O,), float("nan"), dtype=torch.float32, device="cuda")
    qdg.q4_0s_q8_0_gemv(to_dev(Wr), to_dev(xq), y, O, K)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    return to_host(y)


# one segment of 8 blocks (K = 256); ragged last segments (2304, 4352, 6400);
# whole segments (4096, 14336, 32768 = 16 segments, one row slot per CTA);
# row counts below, at and above the SM count and ragged.
SEG_SHAPES = [(1, 256), (300, 256), (37, 2304), (1000, 2048), (152, 4096), (153, 4096), (17, 4352),
              (600, 6400), (4096, 14336), (64, 32768), (3000, 768)]


@pytest.mark.parametrize("O,K", SEG_SHAPES)
def test_repack_matches_oracle_bytes(O, K):
    Wq, _ = problem(O + 5 * K, O, K)
    assert np.array_equal(gpu_repack(Wq, O, K), oracle.repack_q4_0_seg(Wq, K))


@pytest.mark.parametrize("O,K", SEG_SHAPES)
def test_seg_gemv_block_sums_exact(O, K):
    Wq, xq = problem(O * 7 + K, O, K)
    Wr = oracle.repack_q4_0_seg(Wq, K)
    torch = torch_cuda()
    isum = torch.full((1, O, K // 32), -2 ** 31, dtype=torch.int32, device="cuda")
    qdg.qdg_debug_block_sums(to_dev(Wr), to_dev(xq), isum, O, K, 1, 3)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(isum), oracle.block_sums(Wq, xq, K))


@pytest.mark.parametrize("O,K", SEG_SHAPES)
def test_seg_gemv_output_within_tolerance(O, K):
    Wq, xq = problem(O * 11 + K, O, K, outliers=0.01)
    y = gpu_gemv_seg(oracle.repack_q4_0_seg(Wq, K), xq, O, K)
    _, y64, S = oracle.matvec(Wq, xq, K, threads=8)
    assert_within_tol(y[None, :], y64, S)


def test_seg_gemv_special_blocks():
    """All-zero codes -> -8 d_w sum(q_x); all-8 -> 0; all-15 -> 7 d_w sum(q_x)."""
    K, O = 2304, 3
    rng = np.random.default_rng(2)
    xq = oracle.quantize_q8_0(rng.standard_normal((1, K)).astype(np.float32), None)
    W = np.zeros((O, K // 32 * 18), dtype=np.uint8)
    d = np.array([np.float16(0.25).view(np.uint16)], dtype=np.uint16).view(np.uint8)
    for r, byte in enumerate((0x00, 0x88, 0xFF)):
        for b in range(K // 32):
            W[r, b * 18:b * 18 + 2] = d
            W[r, b * 18 + 2:b * 18 + 18] = byte
    y = gpu_gemv_seg(oracle.repack_q4_0_seg(W, K), xq, O, K)
    _, y64, S = oracle.matvec(W, xq, K)
    assert_within_tol(y[None, :], y64, S)
    assert y[1] == 0.0


def test_seg_group_and_concatenation_match_single_calls():
    """q, k, v as a group, and gate + up repacked back to back into one buffer
    and multiplied as one matrix: bit-identical to one call per matrix."""
    torch = torch_cuda()
    K = 4096
    xq = problem(5, 8, K)[1]
    xd = to_dev(xq)
    shapes = {"q": 1024, "k": 256, "v": 256, "gate": 1536, "up": 1536}
    Wq = {n: oracle.quantize_q4_0(synth.weights(9, n, O, K)) for n, O in shapes.items()}
    Wr = {n: to_dev(oracle.repack_q4_0_seg(Wq[n], K)) for n in shapes}
    single = {}
    for n, O in shapes.items():
        y = torch.empty(O, dtype=torch.float32, device="cuda")
        qdg.q4_0s_q8_0_gemv(Wr[n], xd, y, O, K)
        single[n] = y
    ys = [torch.empty(shapes[n], dtype=torch.float32, device="cuda") for n in ("q", "k", "v")]
    qdg.q4_0s_q8_0_gemv_group([Wr[n] for n in ("q", "k", "v")], ys, [shapes[n] for n in ("q", "k", "v")], xd, K)
    # gate and up repacked on the GPU into the two halves of one buffer
    rb = qdg.q4_0_seg_row_bytes(K)
    cat = empty_u8(2 * 1536 * rb)
    qdg.q4_0_repack_seg(to_dev(Wq["gate"]), cat[:1536 * rb], 1536, K)
    qdg.q4_0_repack_seg(to_dev(Wq["up"]), cat[1536 * rb:], 1536, K)
    ycat = torch.empty(3072, dtype=torch.float32, device="cuda")
    qdg.q4_0s_q8_0_gemv(cat, xd, ycat, 3072, K)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    for n, y in zip(("q", "k", "v"), ys):
        assert np.array_equal(to_host(y).view(np.uint32), to_host(single[n]).view(np.uint32)), n
    got = to_host(ycat)
    assert np.array_equal(got[:1536].view(np.uint32), to_host(single["gate"]).view(np.uint32))
    assert np.array_equal(got[1536:].view(np.uint32), to_host(single["up"]).view(np.uint32))
    _, y64, S = oracle.matvec(np.concatenate([Wq["gate"], Wq["up"]]), xq, K, threads=8)
    assert_within_tol(got[None, :], y64, S)


def test_seg_gemv_deterministic_and_pdl_invariant():
    torch = torch_cuda()
    O, K = 4096, 14336
    Wq, xq = problem(78, O, K)
    Wd, xd = to_dev(oracle.repack_q4_0_seg(Wq, K)), to_dev(xq)
    outs = []
    for pdl in (0, 1, 0):
        qdg.qdg_set_option(qdg.QDG_OPT_PDL, pdl)
        y = torch.empty(O, dtype=torch.float32, device="cuda")
        for _ in range(3):
            qdg.q4_0s_q8_0_gemv(Wd, xd, y, O, K)
        torch.cuda.synchronize()
        outs.append(to_host(y))
    qdg.qdg_set_option(qdg.QDG_OPT_PDL, 0)
    assert all(np.array_equal(outs[0].view(np.uint32), o.view(np.uint32)) for o in outs[1:])


def test_seg_gemv_vocab_head_sampled():
    """The 128256 x 4096 vocab head, repacked on the GPU from Q4_0 bytes the
    oracle made, on 2048 sampled rows."""
    torch = torch_cuda()
    O, K = 128256, 4096
    rows = np.sort(synth.sample_indices(O, "head-rows", O, 2048))
    Wq = np.empty((O, K // 32 * 18), dtype=np.uint8)
    for r in range(0, O, 16384):
        r1 = min(O, r + 16384)
        Wq[r:r1] = oracle.quantize_q4_0(synth.weights(3, "head", O, K, row_begin=r, row_end=r1))
    xq = oracle.quantize_q8_0(synth.activations(3, "x", 1, K, outlier_frac=0.01), synth.gamma(3, "g", K), 1e-6)
    Wr = empty_u8(qdg.q4_0_seg_nbytes(O, K))
    qdg.q4_0_repack_seg(to_dev(Wq), Wr, O, K)
    y = torch.empty(O, dtype=torch.float32, device="cuda")
    qdg.q4_0s_q8_0_gemv(Wr, to_dev(xq), y, O, K)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    _, y64, S = oracle.matvec(Wq, xq, K, rows=rows, threads=8)
    assert_within_tol(to_host(y)[rows][None, :], y64, S)


@pytest.mark.parametrize("K", [256, 2304, 4096, 8192, 14336, 16384])
@pytest.mark.parametrize("norm", [True, False])
def test_fused_seg_matches_oracle_and_split(K, norm):
    """The fused form on the segment layout: its Q8_0 vector is the oracle's
    byte for byte, and its outputs equal the split product on that vector bit
    for bit (same kernel arithmetic after the activations)."""
    torch = torch_cuda()
    O = 1000 + K // 8
    seed = K + (7 if norm else 0)
    Wq = oracle.quantize_q4_0(synth.weights(seed, "Wf", O, K))
    x = synth.activations(seed, "xf", 1, K, outlier_frac=0.01)[0]
    gam = synth.gamma(seed, "gf", K) if norm else None
    xq_ref = oracle.quantize_q8_0(x[None, :], gam, 1e-6)
    Wd = to_dev(oracle.repack_q4_0_seg(Wq, K))
    xq_out = empty_u8(qdg.q8_0_nbytes(1, K))
    y = torch.full((O,), float("nan"), dtype=torch.float32, device="cuda")
    qdg.q4_0s_gemv_rmsnorm_group([Wd], [y], [O], to_dev(x), None if gam is None else to_dev(gam), 1e-6, K,
                                 xq_out=xq_out)
    y_split = torch.empty(O, dtype=torch.float32, device="cuda")
    qdg.q4_0s_q8_0_gemv(Wd, to_dev(xq_ref), y_split, O, K)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    assert np.array_equal(to_host(xq_out).reshape(1, -1), xq_ref)
    got = to_host(y)
    assert np.array_equal(got.view(np.uint32), to_host(y_split).view(np.uint32))
    _, y64, S = oracle.matvec(Wq, xq_ref, K, threads=8)
    assert_within_tol(got[None, :], y64, S)


def test_fused_seg_group():
    """q, k, v in one fused launch against the oracle."""
    torch = torch_cuda()
    K = 4096
    shapes = {"q": 4096, "k": 1024, "v": 1024}
    Wq = {n: oracle.quantize_q4_0(synth.weights(12, n, O, K)) for n, O in shapes.items()}
    Wd = [to_dev(oracle.repack_q4_0_seg(Wq[n], K)) for n in shapes]
    x = synth.activations(12, "xg", 1, K, outlier_frac=0.01)[0]
    gam = synth.gamma(12, "gg", K)
    xq_ref = oracle.quantize_q8_0(x[None, :], gam, 1e-6)
    ys = [torch.empty(O, dtype=torch.float32, device="cuda") for O in shapes.values()]
    qdg.q4_0s_gemv_rmsnorm_group(Wd, ys, list(shapes.values()), to_dev(x), to_dev(gam), 1e-6, K)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    for n, y in zip(shapes, ys):
        _, y64, S = oracle.matvec(Wq[n], xq_ref, K, threads=8)
        assert_within_tol(to_host(y)[None, :], y64, S, what=n)


SEG2_SHAPES = [(1, 256), (300, 256), (37, 2304), (1000, 2048), (153, 4096), (17, 4352), (4096, 14336),
               (14336, 4096), (40, 32768)]


@pytest.mark.parametrize("O,K", SEG2_SHAPES)
@pytest.mark.parametrize("N", [2, 3, 4, 8])
def test_seg_small_n_block_sums_exact(O, K, N):
    torch = torch_cuda()
    w = synth.weights(O + 3 * K, "W2", O, K)
    x = synth.activations(O + 3 * K + N, "x2", N, K, outlier_frac=0.01)
    Wq, xq = oracle.quantize_q4_0(w), oracle.quantize_q8_0(x, None)
    isum = torch.full((N, O, K // 32), -2 ** 31, dtype=torch.int32, device="cuda")
    qdg.qdg_debug_block_sums(to_dev(oracle.repack_q4_0_seg(Wq, K)), to_dev(xq), isum, O, K, N, 5)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(isum), oracle.block_sums(Wq, xq, K))


@pytest.mark.parametrize("O,K", SEG2_SHAPES)
@pytest.mark.parametrize("N", [1, 2, 3, 4, 8])
def test_seg_small_n_output_within_tolerance(O, K, N):
    """y [N][ldy] with ldy > O: the padding stays untouched."""
    torch = torch_cuda()
    w = synth.weights(O * 5 + K + N, "W2", O, K)
    x = synth.activations(O * 5 + K + N, "x2", N, K, outlier_frac=0.01)
    gam = synth.gamma(O + K, "g2", K)
    Wq, xq = oracle.quantize_q4_0(w), oracle.quantize_q8_0(x, gam, 1e-6)
    ldy = O + 3
    y = torch.full((N, ldy), float("nan"), dtype=torch.float32, device="cuda")
    qdg.q4_0s_q8_0_gemm_small_n(to_dev(oracle.repack_q4_0_seg(Wq, K)), to_dev(xq), y, ldy, O, K, N)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    got = to_host(y)
    assert np.all(np.isnan(got[:, O:]))
    rows = None if O <= 4096 else synth.sample_indices(O, "rows2", O, 2048)
    _, y64, S = oracle.matvec(Wq, xq, K, rows=rows, threads=8)
    assert_within_tol(got[:, :O] if rows is None else got[:, rows], y64, S)


def test_seg_small_n2_matches_two_single_calls():
    """Each column of the two-vector product equals the one-vector kernel's
    result within the tolerance, and both columns are deterministic."""
    torch = torch_cuda()
    O, K = 14336, 4096
    Wq = oracle.quantize_q4_0(synth.weights(21, "W22", O, K))
    xq = oracle.quantize_q8_0(synth.activations(21, "x22", 2, K, outlier_frac=0.01), None)
    Wd, xd = to_dev(oracle.repack_q4_0_seg(Wq, K)), to_dev(xq)
    y2 = torch.empty((2, O), dtype=torch.float32, device="cuda")
    qdg.q4_0s_q8_0_gemm_small_n(Wd, xd, y2, O, O, K, 2)
    y2b = torch.empty((2, O), dtype=torch.float32, device="cuda")
    qdg.q4_0s_q8_0_gemm_small_n(Wd, xd, y2b, O, O, K, 2)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(y2).view(np.uint32), to_host(y2b).view(np.uint32))
    rows = synth.sample_indices(O, "rows22", O, 1024)
    _, y64, S = oracle.matvec(Wq, xq, K, rows=rows, threads=8)
    assert_within_tol(to_host(y2)[:, rows], y64, S)


@pytest.mark.parametrize("O,K,N", [(14336, 4096, 8), (4096, 14336, 8), (1000, 2048, 5), (37, 2304, 5),
                                   (300, 256, 6), (153, 4096, 7), (40, 32768, 6), (40, 32768, 3),
                                   (33, 16640, 4)])
def test_seg_small_n_mma_matches_plain_layout_kernel(O, K, N):
    """Where the segment layout takes the MMA kernel (N >= 5, or K > 16384)
    it runs the plain-layout kernel's arithmetic in the same order (same
    chunks, same cluster split), so the two agree bit for bit."""
    torch = torch_cuda()
    Wq = oracle.quantize_q4_0(synth.weights(O + K, "W3", O, K))
    xq = oracle.quantize_q8_0(synth.activations(O + K + N, "x3", N, K, outlier_frac=0.01), None)
    ys = torch.full((N, O), float("nan"), dtype=torch.float32, device="cuda")
    yp = torch.full((N, O), float("nan"), dtype=torch.float32, device="cuda")
    xd = to_dev(xq)
    qdg.q4_0s_q8_0_gemm_small_n(to_dev(oracle.repack_q4_0_seg(Wq, K)), xd, ys, O, O, K, N)
    qdg.q4_0_q8_0_gemm_small_n(to_dev(Wq), xd, yp, O, O, K, N)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    assert np.array_equal(to_host(ys).view(np.uint32), to_host(yp).view(np.uint32))


# three and four vectors, K <= 16384: the dp4a kernel with one block a lane
# (half-segments: K = 256 and 2304 have a last half of 8 blocks, 4352 a
# whole-block-free second half, 14336 fourteen halves, 16384 sixteen)
SEGN_SHAPES = [(1, 256), (77, 256), (37, 2304), (17, 4352), (1000, 2048), (153, 4096), (4096, 14336),
               (14336, 4096), (300, 16384), (2500, 8192)]


@pytest.mark.parametrize("O,K", SEGN_SHAPES)
@pytest.mark.parametrize("N", [3, 4])
def test_segn_block_sums_and_outputs(O, K, N):
    """Exact block sums through the test hook, outputs within the tolerance
    (every row up to 4096 rows, 2048 sampled rows beyond), padding of y
    untouched, two launches bit for bit the same, and the launch counted as
    this kernel's."""
    torch = torch_cuda()
    seed = 7 * O + K + N
    Wq = oracle.quantize_q4_0(synth.weights(seed, "Wn", O, K))
    xq = oracle.quantize_q8_0(synth.activations(seed, "xn", N, K, outlier_frac=0.01),
                              synth.gamma(seed, "gn", K), 1e-6)
    Wd, xd = to_dev(oracle.repack_q4_0_seg(Wq, K)), to_dev(xq)
    isum = torch.full((N, O, K // 32), -2 ** 31, dtype=torch.int32, device="cuda")
    qdg.qdg_debug_block_sums(Wd, xd, isum, O, K, N, 5)
    ldy = O + 5
    y = torch.full((N, ldy), float("nan"), dtype=torch.float32, device="cuda")
    y2 = torch.full((N, ldy), float("nan"), dtype=torch.float32, device="cuda")
    before = qdg.qdg_launch_count(13)
    qdg.q4_0s_q8_0_gemm_small_n(Wd, xd, y, ldy, O, K, N)
    qdg.q4_0s_q8_0_gemm_small_n(Wd, xd, y2, ldy, O, K, N)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    assert qdg.qdg_launch_count(13) - before == 2
    rows = None if O <= 4096 else synth.sample_indices(seed, "rowsn", O, 2048)
    ref = oracle.block_sums(Wq if rows is None else Wq[rows], xq, K)
    got_isum = to_host(isum) if rows is None else to_host(isum)[:, rows]
    assert np.array_equal(got_isum, ref)
    got = to_host(y)
    assert np.all(np.isnan(got[:, O:]))
    assert np.array_equal(got.view(np.uint32), to_host(y2).view(np.uint32))
    _, y64, S = oracle.matvec(Wq, xq, K, rows=rows, threads=8)
    assert_within_tol(got[:, :O] if rows is None else got[:, rows], y64, S)


def test_segn_unaligned_activations():
    """A 2-byte aligned vector set (not 16-byte aligned) is read from global
    memory instead of one bulk copy; same results bit for bit."""
    torch = torch_cuda()
    O, K, N = 999, 4096, 4
    Wq = oracle.quantize_q4_0(synth.weights(5, "Wu", O, K))
    xq = oracle.quantize_q8_0(synth.activations(5, "xu", N, K), None)
    Wd = to_dev(oracle.repack_q4_0_seg(Wq, K))
    xa = to_dev(xq)
    buf = torch.zeros(xq.size + 16, dtype=torch.uint8, device="cuda")
    buf[2:2 + xq.size] = xa.reshape(-1)
    xu = buf[2:2 + xq.size]
    ya = torch.empty((N, O), dtype=torch.float32, device="cuda")
    yu = torch.empty((N, O), dtype=torch.float32, device="cuda")
    qdg.q4_0s_q8_0_gemm_small_n(Wd, xa, ya, O, O, K, N)
    qdg.q4_0s_q8_0_gemm_small_n(Wd, xu, yu, O, O, K, N)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    assert np.array_equal(to_host(ya).view(np.uint32), to_host(yu).view(np.uint32))


def raw_q4_0(seed, name, O, K):
    """Seeded random Q4_0 rows (every nibble pattern is a valid block) with a
    fixed finite fp16 scale in every block."""
    W = synth.raw_bytes(seed, name, O * (K // 32) * 18).reshape(O, K // 32, 18)
    W[:, :, 0:2] = np.frombuffer(np.float16(0.004).tobytes(), dtype=np.uint8)
    return W.reshape(O, -1)


@pytest.mark.parametrize("O,K,N", [(29500, 32768, 1), (14800, 32768, 2), (118000, 4096, 2), (7500, 16384, 4),
                                   (9900, 16384, 3)])
def test_seg_rows_in_two_chunks(O, K, N):
    """More rows per CTA than one chunk of partial sums holds, so each CTA
    fills its ring again at the chunk boundary: the batch-1 GEMV at K = 32768
    (192 rows a chunk, 194-195 rows a CTA), the two-vector kernel at K = 32768
    (96 rows a chunk, 97-98 rows a CTA) and at K = 4096 (768 rows a chunk,
    776-777 rows a CTA), and the three/four-vector dp4a
    kernel at K = 16384 (four vectors: 48 rows a chunk, 49-50 rows a CTA;
    three: 64 rows a chunk, 65-66 rows a CTA).  Exact block sums and outputs
    on sampled rows."""
    torch = torch_cuda()
    Wq = raw_q4_0(O + N, "Wchunks", O, K)
    xq = oracle.quantize_q8_0(synth.activations(O + N, "xchunks", N, K, outlier_frac=0.01), None)
    Wd, xd = to_dev(oracle.repack_q4_0_seg(Wq, K)), to_dev(xq)
    rows = synth.sample_indices(O + N, "rows-chunks", O, 384)
    isum = torch.full((N, O, K // 32), -2 ** 31, dtype=torch.int32, device="cuda")
    qdg.qdg_debug_block_sums(Wd, xd, isum, O, K, N, 3 if N == 1 else 5)
    y = torch.full((N, O), float("nan"), dtype=torch.float32, device="cuda")
    if N == 1:
        qdg.q4_0s_q8_0_gemv(Wd, xd, y[0], O, K)
    else:
        qdg.q4_0s_q8_0_gemm_small_n(Wd, xd, y, O, O, K, N)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    assert np.array_equal(to_host(isum)[:, rows], oracle.block_sums(Wq[rows], xq, K))
    _, y64, S = oracle.matvec(Wq, xq, K, rows=rows, threads=8)
    assert_within_tol(to_host(y)[:, rows], y64, S)


def test_fused_seg_rows_in_two_chunks():
    """The fused norm+quantize+GEMV on the segment layout with more rows per
    CTA than one chunk holds (K = 16384: 384 rows a chunk; O = 58400 gives
    384-385 rows a CTA): its Q8_0 vector is the oracle's byte for byte and its
    outputs are within tolerance on sampled rows."""
    torch = torch_cuda()
    O, K = 58400, 16384
    Wq = raw_q4_0(O, "Wfc", O, K)
    x = synth.activations(O, "xfc", 1, K, outlier_frac=0.01)[0]
    gam = synth.gamma(O, "gfc", K)
    xq_ref = oracle.quantize_q8_0(x[None, :], gam, 1e-6)
    Wd = to_dev(oracle.repack_q4_0_seg(Wq, K))
    xq_out = empty_u8(qdg.q8_0_nbytes(1, K))
    y = torch.full((O,), float("nan"), dtype=torch.float32, device="cuda")
    qdg.q4_0s_gemv_rmsnorm_group([Wd], [y], [O], to_dev(x), to_dev(gam), 1e-6, K, xq_out=xq_out)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    assert np.array_equal(to_host(xq_out).reshape(1, -1), xq_ref)
    rows = synth.sample_indices(O, "rows-fc", O, 384)
    _, y64, S = oracle.matvec(Wq, xq_ref, K, rows=rows, threads=8)
    assert_within_tol(to_host(y)[rows][None, :], y64, S)


def test_seg_deep_ring_matches_four_deep():
    """A launch with at least 384 rows per CTA takes the eight-deep ring: one
    launch over 60000 rows (395 a CTA) against the same rows as two launches
    of 30000 (197 a CTA, the four-deep ring).  Per-row arithmetic is the same,
    so the outputs agree bit for bit; sampled rows against the oracle."""
    torch = torch_cuda()
    O, K = 60000, 4096
    Wq = raw_q4_0(O, "Wdeep", O, K)
    xq = oracle.quantize_q8_0(synth.activations(O, "xdeep", 1, K, outlier_frac=0.01), None)
    Wr = oracle.repack_q4_0_seg(Wq, K)
    Wd, xd = to_dev(Wr), to_dev(xq)
    y = torch.full((O,), float("nan"), dtype=torch.float32, device="cuda")
    qdg.q4_0s_q8_0_gemv(Wd, xd, y, O, K)
    h = O // 2
    y2 = torch.full((O,), float("nan"), dtype=torch.float32, device="cuda")
    qdg.q4_0s_q8_0_gemv(Wd[:h], xd, y2[:h], h, K)          # rows [0, h): 16-byte aligned (h x 2304 bytes)
    qdg.q4_0s_q8_0_gemv(Wd[h:], xd, y2[h:], O - h, K)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    assert np.array_equal(to_host(y).view(np.uint32), to_host(y2).view(np.uint32))
    rows = synth.sample_indices(O, "rows-deep", O, 256)
    _, y64, S = oracle.matvec(Wq, xq, K, rows=rows, threads=8)
    assert_within_tol(to_host(y)[rows][None, :], y64, S)
