"""GPU parity of the decode-step chain (q4_0s_gemv_chain): every stage's
Q8_0 vector bit for bit against the oracle's quantizer, every output row
within 1e-5 * sum_b |d_w d_x isum_b| of the oracle's fp64 product.

Cases: ragged and whole last segments (K = 256 .. 16384, units of 4, 2 and 1
rows), row counts that leave a partial last unit, groups of up to four
matrices, the most stages a launch takes, repeated launches and graph
replays on one workspace (its counters left zero by every launch), and a stage
whose input is an earlier stage's output."""
import numpy as np
import pytest

import oracle
from quantized_decode_gemv_rms_gb300 import qdg, synth
from helpers import assert_within_tol, to_dev, to_host, torch_cuda

pytestmark = pytest.mark.gpu

EPS = 1e-6


def make_stage(seed, K, Os, norm, outliers=0.0):
    """Host inputs of one stage and the oracle's expectations."""
    x = synth.activations(seed, "chain-x", 1, K, outlier_frac=outliers)
    gam = synth.gamma(seed, "chain-g", K) if norm else None
    Wq = [oracle.quantize_q4_0(synth.weights(seed, f"chain-W{i}", O, K)) for i, O in enumerate(Os)]
    return {"x": x, "gamma": gam, "K": K, "Wq": Wq, "Os": list(Os)}


def expectations(st):
    xq = oracle.quantize_q8_0(st["x"], st["gamma"], EPS)
    ys = [oracle.matvec(Wq, xq, st["K"], threads=8) for Wq in st["Wq"]]
    return xq, ys


def to_device_stage(st):
    torch = torch_cuda()
    K = st["K"]
    return {"x": to_dev(st["x"][0]), "gamma": None if st["gamma"] is None else to_dev(st["gamma"]), "K": K,
            "Ws": [to_dev(oracle.repack_q4_0_seg(Wq, K)) for Wq in st["Wq"]],
            "ys": [torch.full((O,), float("nan"), dtype=torch.float32, device="cuda") for O in st["Os"]],
            "Os": st["Os"],
            "xq_out": torch.zeros(qdg.q8_0_nbytes(1, K), dtype=torch.uint8, device="cuda")}


def new_workspace():
    torch = torch_cuda()
    return torch.zeros(qdg.q4_0s_gemv_chain_workspace_bytes(), dtype=torch.uint8, device="cuda")


def counters_zero(ws):
    return int(ws[:64].sum()) == 0


def check(dev_stages, host_stages, what=""):
    for g, (d, h) in enumerate(zip(dev_stages, host_stages)):
        xq, ys = expectations(h)
        assert np.array_equal(to_host(d["xq_out"]).reshape(1, -1), xq), f"{what} stage {g}: Q8_0 vector differs"
        for i, (yd, (_, y64, S)) in enumerate(zip(d["ys"], ys)):
            assert_within_tol(to_host(yd)[None, :], y64, S, what=f"{what} stage {g} matrix {i}")


# (K, row counts, norm): ragged last segments (256: one segment of 8 blocks;
# 2304, 8448: last segment of 8 blocks), whole segments (4096, 14336, 16384);
# units of 4 rows (K <= 4096), 2 rows (K = 8192: 4 segments), 1 row (K >= 8448)
STAGE_SHAPES = [
    (256, (1,), True),
    (256, (7, 3, 130, 1), False),
    (2304, (37, 515), True),
    (4096, (152, 153, 5), True),
    (8192, (1031,), False),
    (8448, (77, 2), True),
    (14336, (4096,), False),
    (16384, (333,), True),
]


@pytest.mark.parametrize("K,Os,norm", STAGE_SHAPES)
def test_chain_single_stage(K, Os, norm):
    torch = torch_cuda()
    h = make_stage(K + sum(Os), K, Os, norm, outliers=0.01)
    d = to_device_stage(h)
    ws = new_workspace()
    qdg.q4_0s_gemv_chain([d], EPS, ws)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    check([d], [h], f"K={K}")
    assert counters_zero(ws), "barrier counters not returned to zero"


def test_chain_eight_stages_and_repeats():
    """The most stages one launch takes, three launches in a row and a graph
    of two launches replayed twice on one workspace; every launch gives the
    same bits."""
    torch = torch_cuda()
    shapes = [(4096, (4096, 1024, 1024), True), (4096, (4096,), False), (4096, (2000, 2000), True),
              (14336, (4096,), False), (2048, (300,), True), (256, (64, 64, 64, 64), True),
              (8192, (500,), True), (4096, (6000,), True)]
    hs = [make_stage(100 + g, K, Os, norm) for g, (K, Os, norm) in enumerate(shapes)]
    ds = [to_device_stage(h) for h in hs]
    ws = new_workspace()
    arr = qdg.chain_stages(ds)
    qdg.q4_0s_gemv_chain(arr, EPS, ws)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    check(ds, hs, "8 stages")
    first = [to_host(y).copy() for d in ds for y in d["ys"]]
    for _ in range(2):
        for d in ds:
            for y in d["ys"]:
                y.fill_(float("nan"))
        qdg.q4_0s_gemv_chain(arr, EPS, ws)
        torch.cuda.synchronize()
        again = [to_host(y) for d in ds for y in d["ys"]]
        assert all(np.array_equal(a.view(np.uint32), b.view(np.uint32)) for a, b in zip(first, again))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=side):
            qdg.q4_0s_gemv_chain(arr, EPS, ws)
            qdg.q4_0s_gemv_chain(arr, EPS, ws)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        for d in ds:
            for y in d["ys"]:
                y.fill_(float("nan"))
        gr.replay()
        torch.cuda.synchronize()
        assert qdg.qdg_device_status() == qdg.QDG_OK
        again = [to_host(y) for d in ds for y in d["ys"]]
        assert all(np.array_equal(a.view(np.uint32), b.view(np.uint32)) for a, b in zip(first, again))
    assert counters_zero(ws)


def test_chain_stage_reads_earlier_output():
    """Stage 1's input is stage 0's output (K1 = O0).  Stage 0's weights
    have one block per row with codes other than 8 (the rest contribute
    exactly zero), so each y0 is one exact product d_w d_x isum rounded once
    and the oracle's fp32 y0 is the GPU's bit for bit; the oracle then
    quantizes its own y0 for stage 1."""
    torch = torch_cuda()
    K0, O0, O1 = 2048, 1024, 700
    rng = np.random.Generator(np.random.PCG64(77))
    nb = K0 // 32
    h0 = make_stage(7, K0, (O0,), True)
    Wq = h0["Wq"][0].reshape(O0, nb, 18).copy()
    Wq[:, :, 2:] = 0x88                                  # every code 8: the block contributes exactly 0
    for o in range(O0):
        b = o % nb
        Wq[o, b, 2:] = rng.integers(0, 256, size=16, dtype=np.uint8)
    h0["Wq"][0] = Wq.reshape(O0, -1)
    xq0 = oracle.quantize_q8_0(h0["x"], h0["gamma"], EPS)
    # y0_64 is exact (one block's product, at most 38 significant bits), so
    # y0_32 is that value rounded once, as the kernel rounds its single product
    y0_32, y0_64, S0 = oracle.matvec(h0["Wq"][0], xq0, K0)
    h1 = make_stage(8, O0, (O1,), True)
    h1["x"] = y0_32.astype(np.float32)
    d0 = to_device_stage(h0)
    d1 = to_device_stage(h1)
    d1["x"] = d0["ys"][0]                                 # the chain reads stage 0's output
    ws = new_workspace()
    qdg.q4_0s_gemv_chain([d0, d1], EPS, ws)
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    assert np.array_equal(to_host(d0["ys"][0]).view(np.uint32), y0_32[0].view(np.uint32))
    check([d0, d1], [h0, h1], "aliased")
