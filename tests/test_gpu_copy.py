"""dsa_copy_async: the staging copy by a kernel, between pinned host memory and
device memory and device to device, bit for bit; pageable host memory and
overlapping ranges are refused on the host before any launch."""
import ctypes as C

import numpy as np
import pytest
import torch

import dynamic_sparse_attention_indexer_gb300 as dsa
from dynamic_sparse_attention_indexer_gb300 import _abi

pytestmark = pytest.mark.gpu
INVALID = 1


def _bytes(n, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, 256, (n,), dtype=torch.uint8, generator=g)


@pytest.mark.parametrize("n", [16, 4096, (1 << 20) + 48, 131584])
def test_round_trip_pinned_device_pinned(n):
    dev = torch.device("cuda", 0)
    src = _bytes(n, n).pin_memory()
    mid = torch.empty(n, dtype=torch.uint8, device=dev)
    back = torch.zeros(n, dtype=torch.uint8).pin_memory()
    dsa.copy_async(mid, src)
    dsa.copy_async(back, mid)
    torch.cuda.synchronize()
    assert torch.equal(mid.cpu(), src)
    assert torch.equal(back, src)
    assert dsa.check_device_status(dev) == 0


def test_device_to_device_and_views():
    dev = torch.device("cuda", 0)
    a = _bytes(65536, 7).to(dev)
    b = torch.empty(65536 + 32, dtype=torch.uint8, device=dev)
    dsa.copy_async(b[16:16 + 65536], a)  # a 16-byte aligned view
    torch.cuda.synchronize()
    assert torch.equal(b[16:16 + 65536], a)


def test_refuses_pageable_host_memory_and_overlap():
    lib = _abi.load()
    dev = torch.device("cuda", 0)
    d = torch.empty(4096, dtype=torch.uint8, device=dev)
    host = np.zeros(4096 + 16, dtype=np.uint8)
    p = host.ctypes.data + (-host.ctypes.data % 16)  # pageable, 16-byte aligned
    stream = C.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    assert lib.dsa_copy_async(p, d.data_ptr(), 4096, stream) == INVALID
    assert lib.dsa_copy_async(d.data_ptr(), p, 4096, stream) == INVALID
    assert lib.dsa_copy_async(d.data_ptr() + 1024, d.data_ptr(), 2048, stream) == INVALID
    torch.cuda.synchronize()
    assert dsa.check_device_status(dev) == 0
