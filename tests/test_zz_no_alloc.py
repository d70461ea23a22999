"""nf4_quantize_noalloc: the allocation-free variant of nf4_quantize, for callers that may not
allocate device memory (a fixed, pre-reserved memory budget).  It must give exactly what the
workspace version gives, call after call, although every call reuses the library's one scratch
area.  This file is collected last so that a failure here cannot hide any other test."""
import ctypes

import numpy as np
import pytest
import torch

import bit_nf4_quantized_36_b300 as q
from bit_nf4_quantized_36_b300 import _lib, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_nf4_quantized_36_b300 import build
    build.build()
    return _lib.load()


def _host(qw):
    return [t.cpu().numpy() for t in (qw.codes, qw.scale_codes, qw.scale_scales, qw.scale_offset)]


def test_noalloc_equals_workspace_quantize_on_consecutive_calls(L):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # two calls in a row on the shared scratch area, the second with fewer blocks than the first
    for rows, cols, seed in ((1024, 4096, 11), (300, 320, 12)):
        W = torch.from_numpy(synth.weight(seed, rows, cols, 0.02, outliers="uniform")).cuda()
        ref = q.nf4_quantize(W)
        out = q.empty_nf4(rows, cols)
        st = out.struct()
        assert L.nf4_quantize_noalloc(ctypes.c_void_p(W.data_ptr()), ctypes.byref(st), stream) == 0
        torch.cuda.synchronize()
        q.check_device_error()
        for a, b in zip(_host(out), _host(ref)):
            np.testing.assert_array_equal(a.view(np.uint8), b.view(np.uint8))


def test_noalloc_rejects_matrices_beyond_its_scratch(L):
    # 2^28 + 64 weights: refused before any launch (the pointers are never dereferenced)
    big = _lib.NF4TensorStruct(1, (1 << 28) + 64, 0x10000, 0x20000, 0x30000, 0x40000)
    n0 = L.qlora_launch_count()
    assert L.nf4_quantize_noalloc(ctypes.c_void_p(0x50000), ctypes.byref(big), None) == 2
    assert L.qlora_launch_count() == n0


def test_noalloc_call_allocates_nothing_and_launches_two_kernels(L):
    rows, cols = 512, 2048
    W = torch.from_numpy(synth.weight(13, rows, cols, 0.02)).cuda()
    out = q.empty_nf4(rows, cols)
    q.nf4_quantize_noalloc(W, out)  # warm-up: the first call may load the device module
    torch.cuda.synchronize()
    alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    n0 = L.qlora_launch_count()
    q.nf4_quantize_noalloc(W, out)
    torch.cuda.synchronize()
    q.check_device_error()
    # the absmax/code kernel and the scale double-quantization kernel, nothing else
    assert L.qlora_launch_count() - n0 == 2
    assert torch.cuda.memory_allocated() == alloc0
    # device-wide free memory cannot have dropped (it may rise while the driver reclaims what an
    # earlier process on the device released)
    assert torch.cuda.mem_get_info()[0] >= free0
    ref = q.nf4_quantize(W)
    for a, b in zip(_host(out), _host(ref)):
        np.testing.assert_array_equal(a.view(np.uint8), b.view(np.uint8))


def test_noalloc_wrapper_refuses_output_on_another_device(L):
    W = torch.zeros((64, 64), dtype=torch.float32, device="cuda")
    # one device: an output in host memory stands in for "another device"
    bad = q.empty_nf4(64, 64, device="cpu" if torch.cuda.device_count() < 2 else "cuda:1")
    with pytest.raises(ValueError):
        q.nf4_quantize_noalloc(W, bad)
