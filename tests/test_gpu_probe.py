"""The roofline probe's streaming-copy kernel (hicache_stream_copy): it moves
every byte exactly, in each direction, at sizes that leave ragged tails; and
every argument it refuses is refused on the host, with nothing launched."""
import numpy as np
import pytest
import torch

import tiered_kv_cache_gb300 as hc
from tiered_kv_cache_gb300 import build as hc_build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    hc_build.build()
    torch.cuda.init()


@pytest.mark.parametrize("nbytes,grid,vecs", [(16, 0, 4), (4096 + 48, 3, 8), ((1 << 22) + 16 * 77, 5, 4),
                                              ((64 << 20) - 16, 0, 8)])
def test_stream_copy_moves_every_byte(nbytes, grid, vecs):
    g = torch.Generator(device="cuda")
    g.manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes + 64,), dtype=torch.uint8, device="cuda", generator=g)
    mem = hc.PinnedHost(nbytes + 64)
    host = np.frombuffer((np.ctypeslib.ctypes.c_uint8 * (nbytes + 64)).from_address(mem.ptr), np.uint8)
    host[:] = 0xA5
    c0 = hc.launch_count()
    hc.stream_copy(mem.ptr, src.data_ptr(), nbytes, grid, vecs)           # device -> host
    torch.cuda.synchronize()
    assert hc.launch_count() - c0 == 1
    want = src.cpu().numpy()
    assert np.array_equal(host[:nbytes], want[:nbytes])
    assert (host[nbytes:] == 0xA5).all()
    dst = torch.full((nbytes + 64,), 0x3C, dtype=torch.uint8, device="cuda")
    host[:nbytes] = np.random.default_rng(nbytes).integers(0, 256, nbytes, dtype=np.uint8)
    hc.stream_copy(dst.data_ptr(), mem.ptr, nbytes, grid, vecs)           # host -> device
    torch.cuda.synchronize()
    got = dst.cpu().numpy()
    assert np.array_equal(got[:nbytes], host[:nbytes])
    assert (got[nbytes:] == 0x3C).all()
    dst2 = torch.zeros_like(dst)
    hc.stream_copy(dst2.data_ptr(), dst.data_ptr(), nbytes, grid, vecs)   # device -> device
    torch.cuda.synchronize()
    assert torch.equal(dst2[:nbytes], dst[:nbytes])
    del host
    mem.free()


def test_stream_copy_refusals_launch_nothing():
    dev = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    mem = hc.PinnedHost(1 << 16)
    pageable = np.zeros(1 << 16, np.uint8)
    c0 = hc.launch_count()
    cases = [
        ((dev.data_ptr() + 8, mem.ptr, 1024, 0, 4), "ALIGNMENT"),          # misaligned dst
        ((dev.data_ptr(), mem.ptr, 1000, 0, 4), "ALIGNMENT"),              # not a multiple of 16
        ((dev.data_ptr(), pageable.ctypes.data, 1024, 0, 4), "NOT_PINNED"),  # pageable source
        ((dev.data_ptr(), dev.data_ptr() + 512, 1024, 0, 4), "INVALID_ARG"),  # overlap
        ((dev.data_ptr(), mem.ptr, 1024, 0, 6), "INVALID_ARG"),            # vectors per thread
        ((dev.data_ptr(), mem.ptr, 1024, -2, 4), "INVALID_ARG"),           # grid
        ((0, mem.ptr, 1024, 0, 4), "INVALID_ARG"),                         # NULL
    ]
    for args, status in cases:
        with pytest.raises(hc.HiCacheError) as e:
            hc.stream_copy(*args)
        assert e.value.status == status, (args, e.value)
    hc.stream_copy(dev.data_ptr(), mem.ptr, 0)                             # nothing to do
    assert hc.launch_count() == c0
    mem.free()
