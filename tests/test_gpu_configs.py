"""The two small decode configurations end to end on the GPU, every output
checked against the oracle:

  * the 256 x 256 parity case (seed 0, one vector through RMSNorm*gamma ->
    Q8_0, Q4_0 weights quantized on the GPU), through the split route (the
    quantize kernel, then the GEMV on either weight layout) and the fused
    route (one norm + quantize + GEMV launch on either layout);
  * the Llama-3.2-1B-shaped decode step (hidden 2048, GQA k/v 512, FFN 8192;
    the down projection on a plain-quantized input) through the benchmark's
    own step object, in its launch configuration (a CUDA graph of consecutive
    steps with programmatic dependent launch), on all four routes.

Llama-3.2-1B is one of the two models whose decode speed the OpenVINO
backend page measures [llama.cpp b10981: OpenVINO backend optimises stateful
decode and GPU MoE inference, section "KV state reorder ... 6.27 -> 9.11
t/s"].  Bars: Q8_0 and Q4_0 bytes identical, outputs within 1e-5 * S."""
import numpy as np
import pytest

import bench
import oracle
from quantized_decode_gemv_rms_gb300 import qdg, synth, workloads
from helpers import assert_within_tol, to_dev, to_host, torch_cuda

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------- tiny 256 x 256
def _tiny_inputs():
    wl = workloads.TINY
    (m,) = wl.matrices
    x = synth.activations(wl.seed, "x:x:0", 1, m.cols)
    gam = synth.gamma(wl.seed, "x", m.cols)
    w = synth.weights(wl.seed, m.name, m.rows, m.cols)
    return wl, m, x, gam, w


@pytest.mark.parametrize("route", ["split-plain", "split-seg", "fused-plain", "fused-seg"])
def test_tiny_config(route):
    torch = torch_cuda()
    wl, m, x, gam, w = _tiny_inputs()
    O, K = m.rows, m.cols
    Wq_ref = oracle.quantize_q4_0(w)
    xq_ref = oracle.quantize_q8_0(x, gam, wl.eps)
    _, y64, S = oracle.matvec(Wq_ref, xq_ref, K)

    Wq = torch.empty(qdg.q4_0_nbytes(O, K), dtype=torch.uint8, device="cuda")
    qdg.quantize_q4_0(to_dev(w), Wq)
    Wr = torch.empty(qdg.q4_0_seg_nbytes(O, K), dtype=torch.uint8, device="cuda")
    qdg.q4_0_repack_seg(Wq, Wr, O, K)
    xd, gd = to_dev(x[0]), to_dev(gam)
    xq = torch.zeros(qdg.q8_0_nbytes(1, K), dtype=torch.uint8, device="cuda")
    y = torch.full((O,), float("nan"), dtype=torch.float32, device="cuda")
    if route.startswith("split"):
        qdg.qnorm_quantize_q8_0(xd, gd, wl.eps, xq, K=K, N=1)
        if route.endswith("seg"):
            qdg.q4_0s_q8_0_gemv(Wr, xq, y, O, K)
        else:
            qdg.q4_0_q8_0_gemv(Wq, xq, y, O, K)
    elif route.endswith("seg"):
        qdg.q4_0s_gemv_rmsnorm_group([Wr], [y], [O], xd, gd, wl.eps, K, xq_out=xq)
    else:
        qdg.q4_0_gemv_rmsnorm(Wq, xd, gd, wl.eps, y, O, K, xq_out=xq)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    assert np.array_equal(to_host(Wq).reshape(O, -1), Wq_ref), "Q4_0 weights differ from the oracle"
    assert np.array_equal(to_host(Wr).reshape(O, -1), oracle.repack_q4_0_seg(Wq_ref, K))
    assert np.array_equal(to_host(xq).reshape(1, -1), xq_ref), "Q8_0 activations differ from the oracle"
    assert_within_tol(to_host(y)[None, :], y64, S, what=route)


# ---------------------------------------------------------------- Llama-3.2-1B step
WL1B = workloads.LLAMA_1B


@pytest.fixture(scope="module")
def expected_1b():
    """Oracle outputs of every row of every projection, per input set."""
    kinds = bench.activation_kinds(WL1B)
    Wq = {m.name: oracle.quantize_q4_0(synth.weights(WL1B.seed, m.name, m.rows, m.cols)) for m in WL1B.matrices}
    out = []
    for p in range(bench.N_INPUT_SETS):
        xq = {}
        for tag, K in WL1B.activations.items():
            x = synth.activations(WL1B.seed, f"x:{tag}:{p}", 1, K, outlier_frac=WL1B.outlier_frac)
            gam = synth.gamma(WL1B.seed, tag, K) if kinds[tag] == "norm" else None
            xq[tag] = oracle.quantize_q8_0(x, gam, WL1B.eps)
        ys = {}
        for m in WL1B.matrices:
            _, y64, S = oracle.matvec(Wq[m.name], xq[m.source.split(":", 1)[1]], m.cols, threads=8)
            ys[m.name] = (y64, S)
        out.append((xq, ys))
    return Wq, out


@pytest.fixture(scope="module")
def step1b():
    torch = torch_cuda()
    qdg.qdg_set_option(qdg.QDG_OPT_PDL, 1)
    st = bench.DecodeStep(WL1B, torch.device("cuda", 0), layout="seg")
    yield st
    qdg.qdg_set_option(qdg.QDG_OPT_PDL, 0)
    del st
    torch.cuda.empty_cache()


def test_1b_weights_match_oracle(step1b, expected_1b):
    Wq, _ = expected_1b
    for m in WL1B.matrices:
        assert np.array_equal(to_host(step1b.W[m.name]).reshape(m.rows, -1), Wq[m.name]), m.name
        assert np.array_equal(to_host(step1b.Wr[m.name]).reshape(m.rows, -1),
                              oracle.repack_q4_0_seg(Wq[m.name], m.cols)), m.name


@pytest.mark.parametrize("route", ["chain-seg", "split-seg", "fused-seg", "split-plain", "fused-plain"])
def test_1b_decode_step_every_row(step1b, expected_1b, route):
    """Each input set's step replayed from one graph; after every step all
    outputs (and, on the split and chain routes, the Q8_0 vectors) are checked."""
    torch = torch_cuda()
    _, exp = expected_1b
    r = route.split("-")[0]
    fused = r == "fused"
    step1b.layout = "seg" if route.endswith("-seg") else "plain"
    for p in range(bench.N_INPUT_SETS):
        step1b.run(step1b.x_dev[p], route=r)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graphs = []
    with torch.cuda.stream(side):
        for p in range(bench.N_INPUT_SETS):
            graphs.append(bench.capture(lambda p=p: step1b.run(step1b.x_dev[p], route=r), side))
    torch.cuda.current_stream().wait_stream(side)
    for p in range(bench.N_INPUT_SETS):
        step1b.y_flat.fill_(float("nan"))
        graphs[p].replay()
        torch.cuda.synchronize()
        assert qdg.qdg_device_status() == qdg.QDG_OK
        xq_ref, ys = exp[p]
        for m in WL1B.matrices:
            y64, S = ys[m.name]
            assert_within_tol(to_host(step1b.y[m.name])[None, :], y64, S, what=f"{route}:{m.name}:set{p}")
        if not fused:
            for tag in WL1B.activations:
                assert np.array_equal(to_host(step1b.xq[tag]).reshape(1, -1), xq_ref[tag]), f"{route}:xq:{tag}"
    step1b.layout = "seg"
