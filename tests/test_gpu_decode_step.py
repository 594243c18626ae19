"""The 8B-shaped decode step at full size, in the launch configuration the
benchmark times: a CUDA graph of consecutive steps (one per input set) with
programmatic dependent launch, through the benchmark's own step object.
Sampled rows of every projection (the first and last rows, rows on both sides
of CTA boundaries, and random rows) are compared with the oracle, for the
split and the fused route, each on the plain and on the segment layout, and
for the chain route (one launch per step)."""
import numpy as np
import pytest

import bench
import oracle
from quantized_decode_gemv_rms_gb300 import qdg, synth, workloads
from helpers import assert_within_tol, to_host, torch_cuda

pytestmark = pytest.mark.gpu

WL = workloads.LLAMA_8B


def sample_rows(O, name, grid=152):
    """Rows the oracle evaluates: both ends, both sides of a few CTA row-range
    boundaries, and random rows from three 1024-row chunks."""
    picks = set(range(0, 24)) | set(range(O - 24, O))
    for c in (1, 37, 76, 151):
        r0 = c * O // grid
        picks |= {r0 - 1, r0, r0 + 1}
    chunks = synth.sample_indices(WL.seed, f"chunks:{name}", -(-O // 1024), 3)
    for c in chunks:
        lo = int(c) * 1024
        hi = min(O, lo + 1024)
        picks |= set((lo + synth.sample_indices(WL.seed, f"rows:{name}:{c}", hi - lo, 48)).tolist())
    return np.array(sorted(r for r in picks if 0 <= r < O), dtype=np.int64)


@pytest.fixture(scope="module")
def expected():
    """Oracle outputs for the last input set of a graph (computed once)."""
    p = bench.N_INPUT_SETS - 1
    kinds = bench.activation_kinds(WL)
    xq = {}
    for tag, K in WL.activations.items():
        x = synth.activations(WL.seed, f"x:{tag}:{p}", 1, K, outlier_frac=WL.outlier_frac)
        gam = synth.gamma(WL.seed, tag, K) if kinds[tag] == "norm" else None
        xq[tag] = oracle.quantize_q8_0(x, gam, WL.eps)
    out = {}
    for m in WL.matrices:
        rows = sample_rows(m.rows, m.name)
        Wq = oracle.quantize_q4_0(synth.weight_rows(WL.seed, m.name, m.rows, m.cols, rows))
        _, y64, S = oracle.matvec(Wq, xq[m.source.split(":", 1)[1]], m.cols, threads=8)
        out[m.name] = (rows, y64, S)
    return out


@pytest.fixture(scope="module")
def step8b():
    torch = torch_cuda()
    qdg.qdg_set_option(qdg.QDG_OPT_PDL, 1)
    st = bench.DecodeStep(WL, torch.device("cuda", 0), layout="plain")
    yield st
    qdg.qdg_set_option(qdg.QDG_OPT_PDL, 0)
    del st
    torch.cuda.empty_cache()


@pytest.mark.parametrize("route", ["split-plain", "split-seg", "fused-plain", "fused-seg", "chain-seg"])
def test_decode_step_full_size_sampled(step8b, expected, route):
    torch = torch_cuda()
    r = route.split("-")[0]
    step8b.layout = "seg" if route.endswith("-seg") else "plain"
    for p in range(3):                      # eager warm-up (also sets kernel attributes)
        step8b.run(step8b.x_dev[p], route=r)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        g = bench.capture(lambda: [step8b.run(step8b.x_dev[p], route=r) for p in range(bench.N_INPUT_SETS)],
                          side)
    torch.cuda.current_stream().wait_stream(side)
    for y in step8b.y.values():
        y.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    for m in WL.matrices:
        rows, y64, S = expected[m.name]
        got = to_host(step8b.y[m.name])[rows]
        assert_within_tol(got[None, :], y64, S, what=f"{route}:{m.name}")


@pytest.mark.parametrize("staging,route", [("direct", "split"), ("direct", "chain"), ("kernel", "chain"),
                                           ("engine", "chain"), ("kernel", "fused"), ("direct", "fused")])
def test_decode_step_from_host_buffers(step8b, expected, staging, route):
    """The end-to-end forms the benchmark times: inputs staged in from pinned
    host memory, the step, every output moved out (stored straight into the
    mapped pinned buffer by the GEMVs, or staged out), in one graph with PDL;
    the host copies of the outputs are checked against the oracle."""
    torch = torch_cuda()
    step8b.layout = "seg"
    for p in range(bench.N_INPUT_SETS):
        bench._e2e_step(step8b, None, p, staging=staging, route=route)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        g = bench.capture(lambda: [bench._e2e_step(step8b, None, p, staging=staging, route=route)
                                   for p in range(bench.N_INPUT_SETS)], side)
    torch.cuda.current_stream().wait_stream(side)
    step8b.y_host_flat.fill_(float("nan"))
    step8b.y_flat.fill_(float("nan"))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert qdg.qdg_device_status() == qdg.QDG_OK
    for m in WL.matrices:
        rows, y64, S = expected[m.name]
        got = step8b.y_host[m.name].numpy()[rows]
        assert_within_tol(got[None, :], y64, S, what=f"{staging}:{route}:{m.name}")
