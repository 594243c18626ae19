"""The staging copy kernel (qdg_stage_copy): pinned host -> device, device ->
pinned host and device -> device moves are byte-identical, for sizes from one
16-byte unit to more than the kernel's grid covers in one pass; pointers the
device cannot reach and bad arguments are refused before any launch."""
import numpy as np
import pytest

from quantized_decode_gemv_rms_gb300 import qdg
from helpers import torch_cuda

pytestmark = pytest.mark.gpu

SIZES = [16, 4096 * 4, 120 * 1024 + 48, (1 << 22) + 16, 171_008 * 4]


def _bytes(n, seed):
    torch = torch_cuda()
    rng = np.random.default_rng(seed)
    return torch.from_numpy(rng.integers(0, 256, size=n, dtype=np.uint8))


@pytest.mark.parametrize("nbytes", SIZES)
def test_host_device_host_round_trip(nbytes):
    torch = torch_cuda()
    src = _bytes(nbytes, nbytes).pin_memory()
    dev = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
    back = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    before = qdg.qdg_launch_count(10)
    qdg.qdg_stage_copy(dev, src)
    qdg.qdg_stage_copy(back, dev)
    torch.cuda.synchronize()
    assert qdg.qdg_launch_count(10) - before == 2
    assert torch.equal(dev.cpu(), src)
    assert torch.equal(back, src)


@pytest.mark.parametrize("nbytes", [16, (1 << 22) + 16])
def test_device_to_device(nbytes):
    torch = torch_cuda()
    a = _bytes(nbytes, 7).cuda()
    b = torch.zeros_like(a)
    qdg.qdg_stage_copy(b, a)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_partial_copy_leaves_the_rest():
    torch = torch_cuda()
    src = _bytes(4096, 3).pin_memory()
    dst = torch.full((4096,), 0x5A, dtype=torch.uint8, device="cuda")
    qdg.qdg_stage_copy(dst, src, 1024)
    torch.cuda.synchronize()
    out = dst.cpu()
    assert torch.equal(out[:1024], src[:1024])
    assert bool((out[1024:] == 0x5A).all())


def test_refuses_pageable_host_memory_and_bad_arguments():
    torch = torch_cuda()
    pageable = torch.zeros(4096, dtype=torch.uint8)          # not pinned: the device cannot reach it
    dev = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    before = qdg.qdg_launch_count(10)
    with pytest.raises(qdg.QdgError) as e:
        qdg.qdg_stage_copy(dev, pageable)
    assert e.value.status == qdg.QDG_EINVAL
    with pytest.raises(qdg.QdgError) as e:
        qdg.qdg_stage_copy(dev[16:], dev[:2048], 2048)      # overlapping ranges
    assert e.value.status == qdg.QDG_EINVAL
    with pytest.raises(qdg.QdgError) as e:
        qdg.qdg_stage_copy(dev[1:], dev[2048:], 16)         # misaligned destination
    assert e.value.status == qdg.QDG_EALIGN
    torch.cuda.synchronize()
    assert qdg.qdg_launch_count(10) == before
