"""GPU parity of nf4_quantize / nf4_dequantize with the CPU oracle: bit-exact codes, scale
codes, second-level scales, offset and bf16 weights."""
import numpy as np
import pytest
import torch

import bit_nf4_quantized_36_b300 as q
from bit_nf4_quantized_36_b300 import synth
from gpu_util import assert_nf4_equal, host_bits, nf4_to_host, quantize_on_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_nf4_quantized_36_b300 import build
    build.build()
    yield
    q.check_device_error()


def _check_roundtrip(orc, W):
    rows, cols = W.shape
    qw = quantize_on_gpu(W)
    ref = orc.nf4_quantize(W)
    assert_nf4_equal(nf4_to_host(qw), ref)
    Wh = host_bits(q.nf4_dequantize(qw))
    Wh_ref = orc.nf4_dequantize(ref["packed"], ref["qcode"], ref["c2"], ref["mu"], rows, cols)
    np.testing.assert_array_equal(Wh, Wh_ref)
    return qw, ref


@pytest.mark.parametrize("rows,cols", [(1, 64), (8, 64), (72, 192), (256, 512), (300, 320), (129, 1088)])
def test_small_shapes(orc, rows, cols):
    g = np.random.default_rng(rows * 1000 + cols)
    W = (g.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    _check_roundtrip(orc, W)


def test_degenerate_blocks(orc):
    g = np.random.default_rng(5)
    W = (g.standard_normal((64, 256)) * 0.02).astype(np.float32)
    W[0, :64] = 0.0                      # all-zero block -> code 7, dequantizes to zeros
    W[1, :] = 0.03125                    # constant blocks
    W[2, 64:128] = -1e-30                # tiny denormal-range magnitudes
    W[3, :64] = np.linspace(-1, 1, 64)   # exact level hits / midpoints after scaling
    W[4, 128:192] = 3.0e4                # large magnitudes
    W[5, :] = -W[5, :]
    qw, ref = _check_roundtrip(orc, W)
    codes = qw.codes.cpu().numpy()
    assert np.all(codes[:32] == 0x77)


def test_all_equal_scales(orc):
    # every block has the same absmax: mu is exact, c2 = 0, all scale codes 0
    W = np.tile(np.array([0.5] + [0.1] * 63, np.float32), (40, 4))
    qw, ref = _check_roundtrip(orc, W)
    assert np.all(qw.scale_codes.cpu().numpy() == 0)


def test_scale_mean_tree_order(orc):
    """Block scales (2^53, 2^29 in group 0; 1 in groups 1 and 3; zeros elsewhere) for which the
    pairing order of the mean's tree decides the fp32 mean (2^43 under the oracle's order): the
    GPU's per-group chain and its subtree pairing must land on the same value."""
    W = np.zeros((1, 1024 * 64), np.float32)
    W[0, 0] = 2.0 ** 53
    W[0, 64] = 2.0 ** 29
    W[0, 256 * 64] = 1.0
    W[0, 768 * 64] = 1.0
    qw, ref = _check_roundtrip(orc, W)
    assert float(ref["mu"]) == 2.0 ** 43


def test_tiny_workload(orc):
    _check_roundtrip(orc, synth.tiny_inputs().W)


def test_llama8b_attn_weight(orc):
    W = synth.weight(synth.LLAMA8B_ATTN["id"], 4096, 4096, 0.02)
    _check_roundtrip(orc, W)


def test_llama8b_mlp_weight_with_outliers(orc):
    W = synth.weight(synth.LLAMA8B_MLP["id"], 4096, 14336, 0.02, outliers="uniform", sub=2)
    _check_roundtrip(orc, W)


def test_code_rule_near_every_decision_point(orc):
    """Blocks whose absmax is exactly 1.0, so x = w: every fp32 value within 4096 ulps of each
    midpoint between adjacent levels, plus a strided sweep of all fp32 in [-1, 1]."""
    L = orc.nf4_levels()
    vals = []
    for k in range(15):
        m = np.float32((np.float64(L[k]) + np.float64(L[k + 1])) / 2)
        mb = int(np.array([m], np.float32).view(np.int32)[0])
        bits = np.arange(mb - 4096, mb + 4097, dtype=np.int64)  # 4096 neighbours on each side
        vals.append(bits.astype(np.uint32).view(np.float32))
    pos = np.arange(0, 0x3F800000 + 1, 4099, dtype=np.uint32).view(np.float32)
    vals.append(pos)
    vals.append(-pos)
    v = np.concatenate(vals).astype(np.float32)
    v = v[np.isfinite(v) & (np.abs(v) <= 1.0)]
    # 63 payload values + one 1.0 per block
    nblk = (v.size + 62) // 63
    pad = np.zeros(nblk * 63, np.float32)
    pad[:v.size] = v
    W = np.concatenate([np.ones((nblk, 1), np.float32), pad.reshape(nblk, 63)], axis=1)
    rows = (nblk + 7) // 8 * 8
    Wm = np.zeros((rows, 64), np.float32)
    Wm[:nblk] = W
    Wm[nblk:, 0] = 1.0
    qw = quantize_on_gpu(Wm.reshape(-1, 512))  # same flat order, 8 blocks per row
    got = orc.unpack_nibbles(qw.codes.cpu().numpy())
    want, _ = orc.blockwise_codes(Wm.reshape(-1), 64, L)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("layer,mat", [(0, 0), (39, 4), (79, 1)])
def test_llama70b_sweep_sampled_layers(orc, layer, mat):
    name, rows, cols = synth.LLAMA70B_SWEEP["mats"][mat]
    Wd = synth.sweep_weight_gpu(layer, mat, rows, cols)
    qw = q.nf4_quantize(Wd)
    Wh = q.nf4_dequantize(qw)
    torch.cuda.synchronize()
    W = Wd.cpu().numpy()
    ref = orc.nf4_quantize(W)
    assert_nf4_equal(nf4_to_host(qw), ref)
    Wh_ref = orc.nf4_dequantize(ref["packed"], ref["qcode"], ref["c2"], ref["mu"], rows, cols)
    np.testing.assert_array_equal(host_bits(Wh), Wh_ref)


def test_repeatable(orc):
    W = synth.weight(7, 512, 1024, 0.02)
    a = nf4_to_host(quantize_on_gpu(W))
    b = nf4_to_host(quantize_on_gpu(W))
    assert_nf4_equal(a, b)
