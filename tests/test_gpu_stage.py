"""sv_copy: the device-initiated copy between device memory and page-locked
host memory -- host to device, device to device and device to host, aligned
and misaligned, ragged sizes, bytes around the range untouched, inside a CUDA
graph, and refusal of pageable host memory."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    from speculative_decoding_verification_sv_gb300 import binding
    return binding


@pytest.mark.parametrize("nbytes,off", [(1, 0), (15, 0), (16, 0), (17, 5), (4097, 0), (1000, 3), (70000, 16),
                                        (589056, 0), (3 << 20, 8)])
def test_copy_round_trip(sv, nbytes, off):
    pad = 64
    rng = np.random.default_rng(nbytes + off)
    data = torch.from_numpy(rng.integers(0, 256, nbytes, dtype=np.uint8))
    h_src = torch.zeros(off + nbytes + pad, dtype=torch.uint8).pin_memory()
    h_src[off:off + nbytes] = data
    d1 = torch.full((off + nbytes + pad,), 7, dtype=torch.uint8, device="cuda")
    d2 = torch.full((nbytes + 2 * pad,), 9, dtype=torch.uint8, device="cuda")
    h_dst = torch.full((off + nbytes + pad,), 11, dtype=torch.uint8).pin_memory()
    sv.copy(d1[off:off + nbytes], h_src[off:off + nbytes])     # host -> device
    sv.copy(d2[pad:pad + nbytes], d1[off:off + nbytes])        # device -> device
    sv.copy(h_dst[off:off + nbytes], d2[pad:pad + nbytes])     # device -> host
    torch.cuda.synchronize()
    assert torch.equal(h_dst[off:off + nbytes], data)
    assert torch.equal(d1[off:off + nbytes].cpu(), data)
    # nothing outside the ranges moved
    assert bool((d1[:off] == 7).all()) and bool((d1[off + nbytes:] == 7).all())
    assert bool((d2[:pad] == 9).all()) and bool((d2[pad + nbytes:] == 9).all())
    assert bool((h_dst[:off] == 11).all()) and bool((h_dst[off + nbytes:] == 11).all())


def test_copy_in_a_cuda_graph(sv):
    """The round's shape of use: pinned inputs in, work, result out, captured
    once and replayed with new host data each time."""
    n = 4096
    h_in = torch.zeros(n, dtype=torch.float32).pin_memory()
    h_out = torch.zeros(n, dtype=torch.float32).pin_memory()
    d_in = torch.zeros(n, dtype=torch.float32, device="cuda")
    d_out = torch.zeros(n, dtype=torch.float32, device="cuda")
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        sv.copy(d_in, h_in, stream=st)
        torch.mul(d_in, 2.0, out=d_out)
        sv.copy(h_out, d_out, stream=st)
    for it in range(3):
        vals = torch.arange(n, dtype=torch.float32) + 1000 * it
        h_in.copy_(vals)
        with torch.cuda.stream(st):
            g.replay()
        st.synchronize()
        assert torch.equal(h_out, vals * 2)


def test_copy_refuses_pageable_host_memory(sv):
    d = torch.zeros(64, dtype=torch.uint8, device="cuda")
    h = torch.zeros(64, dtype=torch.uint8)             # pageable
    assert sv.lib.sv_copy(ctypes.c_void_p(d.data_ptr()), ctypes.c_void_p(h.data_ptr()), 64, None) == 1
    assert sv.lib.sv_copy(ctypes.c_void_p(h.data_ptr()), ctypes.c_void_p(d.data_ptr()), 64, None) == 1
    with pytest.raises(ValueError):
        sv.copy(d, h)
    torch.cuda.synchronize()
    assert sv.get_device_error() == 0
