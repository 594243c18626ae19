"""GPU parity of the prefill product (tcgen05 tensor cores) against the CPU
oracle: exact per-block integer sums from the production loop (test hook),
fp32 outputs within 1e-5 * sum_b |d_w d_x isum_b|, full-size prefill shapes
on sampled rows and tokens, ragged tiles, leading dimension, determinism."""
import numpy as np
import pytest

import oracle
from quantized_decode_gemv_rms_gb300 import qdg, synth, workloads
from helpers import assert_within_tol, empty_u8, to_dev, to_host, torch_cuda

pytestmark = pytest.mark.gpu


def problem(seed, O, K, T):
    w = synth.weights(seed, "W", O, K)
    x = synth.activations(seed, "x", T, K)
    return oracle.quantize_q4_0(w), oracle.quantize_q8_0(x, None)


def gpu_gemm(Wd, xd, O, K, T, ldy=None):
    torch = torch_cuda()
    ldy = O if ldy is None else ldy
    y = torch.full((T, ldy), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(qdg.q4_0_q8_0_gemm_workspace_bytes(K, T), dtype=torch.uint8, device="cuda")
    qdg.q4_0_q8_0_gemm(Wd, xd, y, ldy, O, K, T, ws)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    out = to_host(y)
    if ldy > O:
        assert np.all(np.isnan(out[:, O:])), "wrote past O inside the leading dimension"
    return out[:, :O]


SHAPES = [(128, 256, 128), (1, 256, 1), (130, 512, 100), (256, 1024, 256), (300, 2048, 77), (128, 4096, 129),
          (1000, 768, 300)]


@pytest.mark.parametrize("O,K,T", SHAPES)
def test_gemm_block_sums_exact(O, K, T):
    torch = torch_cuda()
    Wq, xq = problem(O + K + T, O, K, T)
    isum = torch.full((T, O, K // 32), -2 ** 31, dtype=torch.int32, device="cuda")
    qdg.qdg_debug_block_sums(to_dev(Wq), to_dev(xq), isum, O, K, T, 2)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    assert np.array_equal(to_host(isum), oracle.block_sums(Wq, xq, K))


@pytest.mark.parametrize("O,K,T", SHAPES)
def test_gemm_output_within_tolerance(O, K, T):
    Wq, xq = problem(O * 3 + K + T, O, K, T)
    y = gpu_gemm(to_dev(Wq), to_dev(xq), O, K, T, ldy=O + 3)
    _, y64, S = oracle.matvec(Wq, xq, K, threads=8)
    assert_within_tol(y, y64, S)


def test_gemm_deterministic():
    O, K, T = 512, 2048, 256
    Wq, xq = problem(9, O, K, T)
    Wd, xd = to_dev(Wq), to_dev(xq)
    a = gpu_gemm(Wd, xd, O, K, T)
    b = gpu_gemm(Wd, xd, O, K, T)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("O,K,T", workloads.PREFILL_SHAPES)
def test_gemm_full_size_sampled(O, K, T):
    """The prefill shapes at full size, with the GPU weight quantizer and the
    fused quantize kernel producing the inputs; sampled rows x sampled tokens
    are recomputed by the oracle from its own quantization of the same data."""
    torch = torch_cuda()
    seed = workloads.PREFILL_SEED
    name = f"prefill-{O}x{K}"
    x = synth.activations(seed, name + "-x", T, K)
    Wq = empty_u8(qdg.q4_0_nbytes(O, K))
    for r in range(0, O, 4096):
        r1 = min(O, r + 4096)
        w = torch.from_numpy(synth.weights(seed, name, O, K, row_begin=r, row_end=r1)).cuda()
        qdg.quantize_q4_0(w, Wq[r * (K // 32) * 18:r1 * (K // 32) * 18], O=r1 - r, K=K)
    xq = empty_u8(qdg.q8_0_nbytes(T, K))
    qdg.qnorm_quantize_q8_0(torch.from_numpy(x).cuda(), None, 0.0, xq)
    y = gpu_gemm(Wq, xq, O, K, T)

    rows = synth.sample_indices(seed, name + "-rows", O, 192)
    toks = synth.sample_indices(seed, name + "-toks", T, 24)
    Wq_ref = oracle.quantize_q4_0(synth.weight_rows(seed, name, O, K, rows))
    xq_ref = oracle.quantize_q8_0(x[toks], None)
    assert np.array_equal(to_host(xq).reshape(T, -1)[toks], xq_ref)
    assert np.array_equal(to_host(Wq).reshape(O, -1)[rows], Wq_ref)
    _, y64, S = oracle.matvec(Wq_ref, xq_ref, K, threads=8)
    assert_within_tol(y[np.ix_(toks, rows)], y64, S)
