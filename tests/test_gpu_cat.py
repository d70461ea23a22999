"""GPU parity of the concatenated projections (qlora_linear_fwd_cat / _bwd_cat) with the oracle:
modules sharing X computed as one N-concatenated layer ("Módulos objetivo": attention
projections, or all linear layers).  Module i's column block of Y must equal its own layer
(oracle layer_fwd_rows); dX is the sum over modules of each module's dX; dA_i, dB_i are each
module's adapter gradients.  Same acceptance as the single-module layer."""
import numpy as np
import pytest
import torch

import bit_nf4_quantized_36_b300 as q
from bit_nf4_quantized_36_b300 import synth
from gpu_util import assert_close, dev_bf16, host_f64, nf4_to_host

pytestmark = pytest.mark.gpu


def _modules(seed, M, K, specs):
    mods = []
    for i, (N, r, alpha) in enumerate(specs):
        mods.append(synth.layer_inputs(seed, M, N, K, r, alpha, sub=i, b_std=0.3))
    X = mods[0].X  # the shared input
    return X, mods


def _oracle_what(orc, W):
    ref = orc.nf4_quantize(W)
    N, K = W.shape
    return ref, orc.nf4_dequantize(ref["packed"], ref["qcode"], ref["c2"], ref["mu"], N, K)


@pytest.mark.parametrize("M,K,specs", [
    (300, 512, [(256, 16, 32.0), (128, 8, 16.0), (128, 5, 10.0)]),   # concatenated path, ragged rank
    (64, 320, [(128, 64, 128.0), (256, 72, 144.0)]),                  # R8 = 136 (3 LoRA k-steps), K % 256 != 0
    (17, 512, [(256, 16, 32.0), (128, 8, 16.0), (128, 5, 10.0)]),    # M <= 32: module by module
    (1, 256, [(128, 4, 8.0), (256, 12, 24.0)]),                       # one token (GEMV per module)
])
def test_cat_matches_each_module(orc, M, K, specs):
    X, mods = _modules(40 + M, M, K, specs)
    dev = torch.device("cuda")
    Xd = dev_bf16(X)
    qws, As, Bs = [], [], []
    for m in mods:
        qws.append(q.nf4_quantize(torch.from_numpy(m.W).to(dev)))
        As.append(dev_bf16(m.A))
        Bs.append(dev_bf16(m.B))
    modules = [(qws[i], As[i], Bs[i], specs[i][2]) for i in range(len(specs))]
    Y, U = q.qlora_linear_fwd_cat(modules, Xd)
    dY = np.concatenate([m.G for m in mods], axis=1)
    dX, dA, dB = q.qlora_linear_bwd_cat(modules, Xd, dev_bf16(dY), U)
    dX2, _, _ = q.qlora_linear_bwd_cat(modules, Xd, dev_bf16(dY), None)  # U recomputed
    torch.cuda.synchronize()
    q.check_device_error()

    Yh, Uh = host_f64(Y), host_f64(U)
    o = c = 0
    dX_ref = np.zeros((M, K))
    for i, (m, (N, r, alpha)) in enumerate(zip(mods, specs)):
        ref, What = _oracle_what(orc, m.W)
        np.testing.assert_array_equal(nf4_to_host(qws[i])["packed"], ref["packed"])
        Yr, Ur = orc.layer_fwd_rows(What, X, m.A, m.B, alpha)
        assert_close(f"Y[{i}]", Yh[:, o:o + N], Yr)
        assert_close(f"U[{i}]", Uh[:, c:c + r], (alpha / r) * Ur)
        assert np.all(Uh[:, c + r:c + (r + 7) // 8 * 8] == 0)
        dX_ref += orc.layer_dx_rows(What, m.A, m.B, m.G, alpha)
        dAr, dBr = orc.layer_adapter_grads(X, m.A, m.B, m.G, alpha)
        assert_close(f"dA[{i}]", dA[i].cpu().numpy(), dAr)
        assert_close(f"dB[{i}]", dB[i].cpu().numpy(), dBr)
        o += N
        c += (r + 7) // 8 * 8
    assert_close("dX", host_f64(dX), dX_ref)
    assert_close("dX (U recomputed)", host_f64(dX2), dX_ref)
