"""Adapter merge on the GPU against the oracle: W_m = bf16(W^ + (alpha/r) B A) ("QLoRA" glossary,
Compromissos: merging needs the base weight dequantized to 16 bits first).  The library forms the
rank-r product in fp32 and rounds fl32(s (B A) + W^) once; the oracle rounds the exact fp64 value
once.  Bar, per element: |W_m - oracle| <= ulp_bf16(oracle) + s r 2^-23 (|B| |A|)[n, k] -- the
two roundings to bf16, plus the worst-case error of an fp32 sum of r terms, which matters only
where W^ and s B A nearly cancel -- and at most 1 % of elements differ at all."""
import numpy as np
import pytest
import torch

import bit_nf4_quantized_36_b300 as q
from bit_nf4_quantized_36_b300 import synth

from gpu_util import host_bits as to_np_u16

pytestmark = pytest.mark.gpu


def _ordinal(bits):
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def _inputs(seed, N, K, r, w_std=0.02, b_std=0.02):
    g = np.random.default_rng(seed)
    W = (g.standard_normal((N, K)) * w_std).astype(np.float32)
    A = (g.standard_normal((r, K)) / np.sqrt(K)).astype(np.float32)
    B = (g.standard_normal((N, r)) * b_std).astype(np.float32)
    return W, A, B


def _run(W, A, B, alpha):
    dev = torch.device("cuda")
    qw = q.nf4_quantize(torch.from_numpy(W).to(dev))
    Ab = torch.from_numpy(A).to(dev).to(torch.bfloat16)
    Bb = torch.from_numpy(B).to(dev).to(torch.bfloat16)
    Wm = q.qlora_merge(qw, Ab, Bb, alpha)
    What = q.nf4_dequantize(qw)
    torch.cuda.synchronize()
    q.check_device_error()
    return qw, to_np_u16(Ab), to_np_u16(Bb), to_np_u16(Wm), to_np_u16(What)


def _f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _ulp_bf16(x):
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return np.exp2(e - 7)


def _check(orc, What, A, B, Wm, alpha, rows=None):
    ref = orc.merge(What if rows is None else What[rows], A, B if rows is None else B[rows], alpha)
    got = Wm if rows is None else Wm[rows]
    Bs = B if rows is None else B[rows]
    r = A.shape[0]
    bound = _ulp_bf16(_f64(ref)) + (alpha / r) * r * 2.0 ** -23 * (np.abs(_f64(Bs)) @ np.abs(_f64(A)))
    diff = np.abs(_f64(got) - _f64(ref))
    worst = np.argmax(diff - bound)
    assert np.all(diff <= bound), f"element {np.unravel_index(worst, diff.shape)}: diff {diff.flat[worst]} > {bound.flat[worst]}"
    off = (got != ref).mean()
    assert off <= 0.01, f"{off:.4f} of elements differ"
    assert np.abs(_ordinal(got) - _ordinal(ref)).max() <= 2


@pytest.mark.parametrize("N,K,r,alpha", [
    (8, 64, 1, 2.0),          # smallest
    (136, 320, 5, 10.0),      # ragged rows and columns, r % 8 != 0 (padded B)
    (256, 512, 16, 32.0),
    (200, 1024, 64, 128.0),   # one full rank chunk
    (128, 256, 72, 16.0),     # two rank chunks, the second ragged
    (64, 768, 256, 512.0),    # maximum rank
])
def test_merge_shapes(orc, N, K, r, alpha):
    W, A, B = _inputs(1000 + r, N, K, r)
    _, Ab, Bb, Wm, What = _run(W, A, B, alpha)
    _check(orc, What, Ab, Bb, Wm, alpha)


def test_merge_zero_adapter_is_the_dequantized_weight():
    W, A, B = _inputs(5, 256, 512, 16)
    _, _, _, Wm, What = _run(W, A, np.zeros_like(B), 32.0)
    assert np.array_equal(Wm, What)


def test_merge_deterministic():
    W, A, B = _inputs(6, 384, 1024, 16)
    dev = torch.device("cuda")
    qw = q.nf4_quantize(torch.from_numpy(W).to(dev))
    Ab = torch.from_numpy(A).to(dev).to(torch.bfloat16)
    Bb = torch.from_numpy(B).to(dev).to(torch.bfloat16)
    a = q.qlora_merge(qw, Ab, Bb, 32.0).clone()
    b = q.qlora_merge(qw, Ab, Bb, 32.0)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_merge_llama70b_up_sampled_rows(orc):
    """28672 x 8192 (the 70B MLP up projection), r = 16, alpha = 32: 64 sampled rows against the
    oracle, at the bench's size and launch configuration."""
    N, K, r = 28672, 8192, 16
    dev = torch.device("cuda")
    W = synth.sweep_weight_gpu(0, 4, N, K)
    qw = q.nf4_quantize(W)
    g = np.random.default_rng(9)
    Ab = torch.from_numpy((g.standard_normal((r, K)) / np.sqrt(K)).astype(np.float32)).to(dev).to(torch.bfloat16)
    Bb = torch.from_numpy((g.standard_normal((N, r)) * 0.01).astype(np.float32)).to(dev).to(torch.bfloat16)
    Wm = q.qlora_merge(qw, Ab, Bb, 32.0)
    What = q.nf4_dequantize(qw)
    torch.cuda.synchronize()
    q.check_device_error()
    rows = np.sort(g.choice(N, 64, replace=False))
    _check(orc, to_np_u16(What)[rows], to_np_u16(Ab), to_np_u16(Bb)[rows], to_np_u16(Wm)[rows], 32.0)
