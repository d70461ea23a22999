"""GPU parity of the layer with LoRA dropout on the adapter input (qlora_linear_fwd_dropout /
_bwd_dropout) against the oracle ("LoRA y QLoRA ..." (coddykit), LoraConfig lora_dropout).
The mask is Philox4x32-10 on both sides (each implemented from the generator's definition), so
the kept elements agree exactly; the layer outputs use the layer's tolerance."""
import numpy as np
import pytest
import torch

import bit_nf4_quantized_36_b300 as q
from bit_nf4_quantized_36_b300 import synth
from gpu_util import assert_close, dev_bf16, host_bits, host_f64

pytestmark = pytest.mark.gpu


def _what(orc, W):
    ref = orc.nf4_quantize(W)
    N, K = W.shape
    return orc.nf4_dequantize(ref["packed"], ref["qcode"], ref["c2"], ref["mu"], N, K)


def test_dropout_mask_is_the_generators(orc):
    """K = r = 64, A = I, s = 1: U = bf16(X_d) element for element, which exposes the mask."""
    M, N, K, r, p, seed, offset = 40, 128, 64, 64, 0.3, 0xDEADBEEF12345678, 5
    inp = synth.layer_inputs(60, M, N, K, r, 64.0)
    A = np.zeros((r, K), dtype=np.uint16)
    A[np.arange(r), np.arange(r)] = 0x3F80
    qw = q.nf4_quantize(torch.from_numpy(inp.W).cuda())
    _, U = q.qlora_linear_fwd_dropout(qw, dev_bf16(inp.X), dev_bf16(A), dev_bf16(inp.B), 64.0, p, seed, offset)
    torch.cuda.synchronize()
    q.check_device_error()
    Ub = host_bits(U)
    D = orc.dropout_scale(seed, offset, p, M, K)
    inv = np.float32(1.0) / (np.float32(1.0) - np.float32(p))
    xf = (inp.X.astype(np.uint32) << 16).view(np.float32)
    want = np.array([orc.bf16_round(float(np.float32(x) * inv)) for x in xf.ravel()], dtype=np.uint16).reshape(M, K)
    want[D == 0] = 0
    np.testing.assert_array_equal(Ub, want)
    assert (D == 0).mean() == pytest.approx(p, abs=0.06)


@pytest.mark.parametrize("M,N,K,r,p", [
    (5, 264, 4160, 8, 0.1),      # the one-launch GEMV (masked X for the adapter term only)
    (17, 256, 512, 8, 0.05),     # small-M kernel
    (300, 264, 320, 24, 0.5),    # CTA pairs, one token tile, ragged
    (600, 256, 512, 16, 0.1),    # CTA pairs, two token tiles
])
def test_dropout_layer_parity(orc, M, N, K, r, p):
    seed, offset = 1000 + M, 3
    inp = synth.layer_inputs(61, M, N, K, r, 2.0 * r, b_std=0.3)
    qw = q.nf4_quantize(torch.from_numpy(inp.W).cuda())
    X, A, B, G = dev_bf16(inp.X), dev_bf16(inp.A), dev_bf16(inp.B), dev_bf16(inp.G)
    Y, U = q.qlora_linear_fwd_dropout(qw, X, A, B, inp.alpha, p, seed, offset)
    dX, dA, dB = q.qlora_linear_bwd_dropout(qw, X, A, B, inp.alpha, p, seed, G, U, offset)
    dX2, dA2, dB2 = q.qlora_linear_bwd_dropout(qw, X, A, B, inp.alpha, p, seed, G, None, offset)
    torch.cuda.synchronize()
    q.check_device_error()
    What = _what(orc, inp.W)
    D = orc.dropout_scale(seed, offset, p, M, K)
    Yr, Ur = orc.layer_fwd_rows_drop(What, inp.X, inp.A, inp.B, inp.alpha, D)
    assert_close("Y", host_f64(Y), Yr)
    assert_close("U", host_f64(U), (inp.alpha / r) * Ur)
    dXr = orc.layer_dx_rows_drop(What, inp.A, inp.B, inp.G, inp.alpha, D)
    dAr, dBr = orc.layer_adapter_grads_drop(inp.X, inp.A, inp.B, inp.G, inp.alpha, D)
    assert_close("dX", host_f64(dX), dXr)
    assert_close("dA", dA.cpu().numpy(), dAr)
    assert_close("dB", dB.cpu().numpy(), dBr)
    # U recomputed in the backward from the regenerated mask: the same values
    assert torch.equal(dX, dX2) and torch.equal(dA, dA2) and torch.equal(dB, dB2)


def test_dropout_p0_is_the_plain_layer():
    inp = synth.layer_inputs(62, 300, 256, 512, 16, 32.0, b_std=0.3)
    qw = q.nf4_quantize(torch.from_numpy(inp.W).cuda())
    X, A, B, G = dev_bf16(inp.X), dev_bf16(inp.A), dev_bf16(inp.B), dev_bf16(inp.G)
    Y0, U0 = q.qlora_linear_fwd(qw, X, A, B, inp.alpha)
    Y1, U1 = q.qlora_linear_fwd_dropout(qw, X, A, B, inp.alpha, 0.0, 7)
    dX0, dA0, dB0 = q.qlora_linear_bwd(qw, X, A, B, inp.alpha, G, U0)
    dX1, dA1, dB1 = q.qlora_linear_bwd_dropout(qw, X, A, B, inp.alpha, 0.0, 7, G, U1)
    torch.cuda.synchronize()
    assert torch.equal(Y0, Y1) and torch.equal(U0, U1)   # the same kernels on the same values
    assert torch.equal(dA0, dA1) and torch.equal(dB0, dB1)
    assert_close("dX", host_f64(dX1), host_f64(dX0))     # dX is formed in two steps under dropout
