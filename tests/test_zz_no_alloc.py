"""The allocation-free prefill entry point (library-owned static scratch)
against the workspace entry point, through the C ABI, on two calls in a row.

Some callers cannot allocate device memory (a plug-in whose host program owns
the GPU's memory through its own pool, code running where cudaMalloc is not
allowed); q4_0_q8_0_gemm_static serves them from a fixed 16 MiB array.  It
runs the same two kernels as the workspace entry on the same records, so its
output must be identical bit for bit.  Collected last; runs alone in a fresh
process as well."""
import numpy as np
import pytest

import oracle
from quantized_decode_gemv_rms_gb300 import qdg, synth
from helpers import assert_within_tol, to_dev, to_host, torch_cuda

pytestmark = pytest.mark.gpu

STATIC_BYTES = 16 << 20


def _problem(seed, O, K, T):
    w = synth.weights(seed, "W", O, K)
    x = synth.activations(seed, "x", T, K, outlier_frac=0.01)
    return oracle.quantize_q4_0(w), oracle.quantize_q8_0(x, None)


# (64, 4096, 1920) is the largest token count the 16 MiB scratch holds at K = 4096
@pytest.mark.parametrize("O,K,T", [(300, 1024, 77), (256, 4096, 200), (64, 4096, 1920)])
def test_static_scratch_matches_workspace_entry(O, K, T):
    torch = torch_cuda()
    assert qdg.q4_0_q8_0_gemm_workspace_bytes(K, T) <= STATIC_BYTES
    Wq, xq = _problem(O + K + T, O, K, T)
    Wd, xd = to_dev(Wq), to_dev(xq)
    ws = torch.empty(qdg.q4_0_q8_0_gemm_workspace_bytes(K, T), dtype=torch.uint8, device="cuda")
    ref = torch.empty((T, O), dtype=torch.float32, device="cuda")
    qdg.q4_0_q8_0_gemm(Wd, xd, ref, O, O, K, T, ws)
    torch.cuda.synchronize()
    ref = to_host(ref)
    _, y64, S = oracle.matvec(Wq, xq, K, threads=8)
    assert_within_tol(ref, y64, S)
    for _ in range(2):   # two calls in a row share the static scratch
        y = torch.full((T, O), float("nan"), dtype=torch.float32, device="cuda")
        qdg.q4_0_q8_0_gemm_static(Wd, xd, y, O, O, K, T)
        torch.cuda.synchronize()
        assert qdg.qdg_device_status() == qdg.QDG_OK
        got = to_host(y)
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), \
            "static-scratch result differs from the workspace entry"


@pytest.mark.parametrize("K,T", [(14336, 640), (4096, 1921)])
def test_static_scratch_rejects_problems_beyond_its_maximum(K, T):
    torch = torch_cuda()
    assert qdg.q4_0_q8_0_gemm_workspace_bytes(K, T) > STATIC_BYTES
    y = torch.empty(1, dtype=torch.float32, device="cuda")
    rc = qdg.lib().q4_0_q8_0_gemm_static(y.data_ptr(), y.data_ptr(), y.data_ptr(), 8, 8, K, T, None)
    assert rc == qdg.QDG_ESHAPE
