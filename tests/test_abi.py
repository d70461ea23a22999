"""The C-ABI library loads, exports every function include/qlora.h declares, and rejects bad
arguments on the host before touching a GPU.  CPU only (no kernel is launched)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

import bit_nf4_quantized_36_b300 as q
from bit_nf4_quantized_36_b300 import _lib, build


@pytest.fixture(scope="module")
def L():
    build.build()
    return _lib.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "qlora.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b([a-z_0-9]+)\s*\([^;{]*\)\s*;", src))


def test_exports_every_declared_symbol(L):
    decl = _declared()
    assert {"nf4_quantize", "nf4_dequantize", "qlora_linear_fwd", "qlora_linear_bwd"} <= decl
    assert decl == set(_lib.EXPORTS)
    for name in decl:
        assert hasattr(L, name), name


def test_status_strings(L):
    for code in range(7):
        assert L.qlora_status_string(code)
    assert L.qlora_status_string(99) == b"unknown status"


def test_storage_bytes_closed_form(L):
    # 4 + 8/64 + 32/(64*256) bits per weight plus the 4-byte offset
    for rows, cols in [(256, 512), (4096, 4096), (8192, 28672), (3, 64)]:
        n = rows * cols
        nb = n // 64
        assert L.qlora_nf4_storage_bytes(rows, cols) == n // 2 + nb + 4 * ((nb + 255) // 256) + 4
    assert L.qlora_nf4_storage_bytes(4, 32) == 0      # cols not a multiple of 64
    assert q.nf4_storage_bytes(4096, 4096) * 8 / (4096 * 4096) == pytest.approx(4.127, abs=1e-3)


def test_workspace_queries(L):
    bad = ctypes.c_size_t(-1).value
    assert L.qlora_quantize_workspace_bytes(4096, 4096) >= 262144 * 4
    assert L.qlora_quantize_workspace_bytes(4, 100) == bad
    for M, N, K, r in [(1, 8, 64, 1), (4096, 4096, 4096, 16), (8192, 14336, 4096, 64), (32, 8192, 28672, 16)]:
        f = L.qlora_fwd_workspace_bytes(M, N, K, r)
        b = L.qlora_bwd_workspace_bytes(M, N, K, r)
        r8 = (r + 7) // 8 * 8
        # U [M, r8] bf16, plus (M > 32, where the scales are rebuilt once per call) fp32 block
        # scales; the backward adds V
        scales = (K // 64) * N * 4 if M > 32 else 0
        assert f >= scales + M * r8 * 2
        assert b >= scales + 2 * M * r8 * 2
    # dropout: the masked input (and, backward, its bits) on top of the plain layer's workspace
    assert L.qlora_fwd_dropout_workspace_bytes(64, 256, 512, 8) >= L.qlora_fwd_workspace_bytes(64, 256, 512, 8) + 64 * 512 * 2
    assert L.qlora_bwd_dropout_workspace_bytes(64, 256, 512, 8) >= L.qlora_bwd_workspace_bytes(64, 256, 512, 8) + 64 * 512 * 2
    assert L.qlora_merge_workspace_bytes(4096, 4096, 16) == 0     # B used in place
    assert L.qlora_merge_workspace_bytes(4096, 4096, 5) >= 4096 * 8 * 2
    assert L.qlora_merge_workspace_bytes(4096, 100, 16) == bad
    assert L.qlora_merge_workspace_bytes(4096, 4096, 0) == bad
    assert L.qlora_fwd_workspace_bytes(16, 256, 100, 8) == bad    # K % 64
    assert L.qlora_fwd_workspace_bytes(16, 250, 512, 8) == bad    # N % 8
    assert L.qlora_fwd_workspace_bytes(16, 256, 512, 0) == bad    # r
    assert L.qlora_fwd_workspace_bytes(16, 256, 512, 257) == bad


def _tensor(rows=256, cols=512, base=0x10000):
    return _lib.NF4TensorStruct(rows, cols, base, base + 0x100000, base + 0x200000, base + 0x300000)


def test_argument_errors_before_any_launch(L):
    P = ctypes.c_void_p
    t = _tensor()
    ws = P(0x40000)
    # NULL weights / tensor
    assert L.nf4_quantize(None, ctypes.byref(t), ws, 1 << 30, None) == 1
    assert L.nf4_quantize(P(0x1000), None, ws, 1 << 30, None) == 1
    # unsupported shapes
    t_bad = _tensor(cols=100)
    assert L.nf4_quantize(P(0x1000), ctypes.byref(t_bad), ws, 1 << 30, None) == 2
    t_empty = _tensor(rows=0)
    assert L.nf4_dequantize(ctypes.byref(t_empty), P(0x1000), None) == 2
    # misaligned pointers
    assert L.nf4_quantize(P(0x1004), ctypes.byref(t), ws, 1 << 30, None) == 3
    t_mis = _lib.NF4TensorStruct(256, 512, 0x10008, 0x20000, 0x30000, 0x40000)
    assert L.nf4_dequantize(ctypes.byref(t_mis), P(0x1000), None) == 3
    # workspace missing / too small
    assert L.nf4_quantize(P(0x1000), ctypes.byref(t), None, 0, None) == 4
    assert L.nf4_quantize(P(0x1000), ctypes.byref(t), ws, 16, None) == 4
    # layer: rank, alpha, N % 8, M
    X, A, B, Y = P(0x1000), P(0x2000), P(0x3000), P(0x4000)
    assert L.qlora_linear_fwd(ctypes.byref(t), X, 16, A, B, 0, 16.0, Y, None, ws, 1 << 30, None) == 1
    assert L.qlora_linear_fwd(ctypes.byref(t), X, 16, A, B, 8, float("nan"), Y, None, ws, 1 << 30, None) == 1
    assert L.qlora_linear_fwd(ctypes.byref(t), X, 0, A, B, 8, 16.0, Y, None, ws, 1 << 30, None) == 2
    t_n = _tensor(rows=250)
    assert L.qlora_linear_fwd(ctypes.byref(t_n), X, 16, A, B, 8, 16.0, Y, None, ws, 1 << 30, None) == 2
    assert L.qlora_linear_fwd(ctypes.byref(t), X, 16, A, B, 8, 16.0, None, None, ws, 1 << 30, None) == 1
    assert L.qlora_linear_fwd(ctypes.byref(t), X, 16, A, B, 8, 16.0, Y, None, ws, 64, None) == 4
    assert L.qlora_linear_bwd(ctypes.byref(t), X, 16, A, B, 8, 16.0, None, None, P(0x5000), P(0x6000),
                              P(0x7000), ws, 1 << 30, None) == 1
    assert L.qlora_linear_bwd(ctypes.byref(t), X, 16, A, B, 8, 16.0, P(0x8008), None, P(0x5000), P(0x6000),
                              P(0x7000), ws, 1 << 30, None) == 3
    # merge: rank, alpha, NULLs, alignment, workspace (needed only when r % 8 != 0)
    Wo = P(0x9000)
    assert L.qlora_merge(ctypes.byref(t), A, B, 0, 16.0, Wo, None, 0, None) == 1
    assert L.qlora_merge(ctypes.byref(t), A, B, 257, 16.0, Wo, None, 0, None) == 1
    assert L.qlora_merge(ctypes.byref(t), A, B, 8, float("inf"), Wo, None, 0, None) == 1
    assert L.qlora_merge(ctypes.byref(t), None, B, 8, 16.0, Wo, None, 0, None) == 1
    assert L.qlora_merge(ctypes.byref(t), A, B, 8, 16.0, None, None, 0, None) == 1
    assert L.qlora_merge(ctypes.byref(t), A, B, 8, 16.0, P(0x9002), None, 0, None) == 3
    assert L.qlora_merge(ctypes.byref(t), A, P(0x3002), 8, 16.0, Wo, None, 0, None) == 3
    assert L.qlora_merge(ctypes.byref(t), A, B, 5, 16.0, Wo, None, 0, None) == 4
    assert L.qlora_merge(ctypes.byref(t), A, B, 5, 16.0, Wo, ws, 64, None) == 4
    # dropout: probability outside [0, 1), missing options
    d_bad = _lib.DropoutStruct(1.0, 1, 0)
    assert L.qlora_linear_fwd_dropout(ctypes.byref(t), X, 16, A, B, 8, 16.0, ctypes.byref(d_bad), Y, None, ws,
                                      1 << 30, None) == 1
    assert L.qlora_linear_fwd_dropout(ctypes.byref(t), X, 16, A, B, 8, 16.0, None, Y, None, ws, 1 << 30, None) == 1
    d_nan = _lib.DropoutStruct(float("nan"), 1, 0)
    assert L.qlora_linear_bwd_dropout(ctypes.byref(t), X, 16, A, B, 8, 16.0, ctypes.byref(d_nan), P(0x8000), None,
                                      P(0x5000), P(0x6000), P(0x7000), ws, 1 << 30, None) == 1
    # AdamW: hyper-parameters out of range, step count, NULL arrays, alignment
    hp = _lib.AdamWStruct(2e-4, 0.9, 0.999, 1e-8, 0.01)
    pa, ga, ma, va = P(0x1000), P(0x2000), P(0x3000), P(0x4000)
    assert L.qlora_adamw_step(None, 1, 16, pa, ga, ma, va, None, None) == 1
    assert L.qlora_adamw_step(ctypes.byref(hp), 0, 16, pa, ga, ma, va, None, None) == 1
    assert L.qlora_adamw_step(ctypes.byref(hp), 1, -1, pa, ga, ma, va, None, None) == 1
    assert L.qlora_adamw_step(ctypes.byref(hp), 1, 0, None, None, None, None, None, None) == 0   # empty: no-op
    for bad in [_lib.AdamWStruct(-1.0, 0.9, 0.999, 1e-8, 0.0), _lib.AdamWStruct(1e-3, 1.0, 0.999, 1e-8, 0.0),
                _lib.AdamWStruct(1e-3, 0.9, float("nan"), 1e-8, 0.0), _lib.AdamWStruct(1e-3, 0.9, 0.999, 0.0, 0.0),
                _lib.AdamWStruct(1e-3, 0.9, 0.999, 1e-8, float("inf"))]:
        assert L.qlora_adamw_step(ctypes.byref(bad), 1, 16, pa, ga, ma, va, None, None) == 1
    assert L.qlora_adamw_step(ctypes.byref(hp), 1, 16, pa, None, ma, va, None, None) == 1
    assert L.qlora_adamw_step(ctypes.byref(hp), 1, 16, P(0x1004), ga, ma, va, None, None) == 3
    assert L.qlora_adamw_step(ctypes.byref(hp), 1, 16, pa, ga, ma, va, P(0x5002), None) == 3
    # paged memory: empty or NULL requests
    out = ctypes.c_void_p(0x1234)
    assert L.qlora_paged_alloc(0, ctypes.byref(out)) == 1 and not out.value
    assert L.qlora_paged_alloc(64, None) == 1
    assert L.qlora_paged_free(None) == 0
    assert L.qlora_paged_prefetch(None, 64, 0, None) == 1
    assert L.qlora_paged_prefetch(P(0x1000), 64, -2, None) == 1
    # failure-path test hook: unknown flags are refused before the device is touched
    assert L.qlora_test_inject(2) == 1 and L.qlora_test_inject(0xFFFFFFFF) == 1
    assert L.qlora_launch_count() == 0  # nothing above reached a kernel launch


def test_library_levels_match_the_format_definition(L):
    # the kernels' constants must be the NF4 table of the glossary snippet (checked here against
    # statistics.NormalDist, independently of the oracle)
    import statistics
    import numpy as np
    nd = statistics.NormalDist()
    top = 0.9677083
    v = sorted([-nd.inv_cdf(top + (0.5 - top) * j / 7) for j in range(7)] + [0.0]
               + [nd.inv_cdf(top + (0.5 - top) * i / 8) for i in range(8)])
    want = np.array([x / v[-1] for x in v], dtype=np.float32)
    got = q.nf4_levels().numpy()
    assert got.view(np.uint32).tolist() == want.view(np.uint32).tolist()


def test_product_path_has_no_fallback(tmp_path, monkeypatch):
    # with the library missing, the binding raises instead of computing anything itself
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        q.launch_count()
