"""The seeded input recipe (bit_nf4_quantized_36_b300/synth.py) checked against its own
statement: shapes, distributions, outlier rates, bf16 rounding and repeatability.  These are the
inputs every parity test and the benchmark use, so a drift here would silently change what is
measured."""
import math

import numpy as np
import pytest

from bit_nf4_quantized_36_b300 import synth


def _bf16_rne(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even fp32 -> bf16 bits, written out on the integer bit pattern (finite
    inputs): an implementation independent of the torch cast synth uses."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def _bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _std_ok(x, want, n):
    # sample std of n normal draws: relative standard error ~ 1/sqrt(2n); allow 6 of them
    return abs(np.std(x) / want - 1.0) < 6.0 / math.sqrt(2.0 * n)


def test_repeatable_and_distinct_streams():
    a = synth.layer_inputs(900, 32, 128, 256, 8, 16.0)
    b = synth.layer_inputs(900, 32, 128, 256, 8, 16.0)
    c = synth.layer_inputs(900, 32, 128, 256, 8, 16.0, sub=1)
    for k in ("W", "X", "A", "B", "G"):
        np.testing.assert_array_equal(getattr(a, k), getattr(b, k))
        assert not np.array_equal(getattr(a, k), getattr(c, k)), k
    # tensors of one workload come from different streams
    assert not np.array_equal(a.X[:, :128], a.G[:, :128])


def test_layer_inputs_shapes_and_distributions():
    M, N, K, r = 512, 1024, 2048, 16
    inp = synth.layer_inputs(901, M, N, K, r, 32.0)
    assert inp.W.dtype == np.float32 and inp.W.shape == (N, K)
    for k, shape in (("X", (M, K)), ("A", (r, K)), ("B", (N, r)), ("G", (M, N))):
        t = getattr(inp, k)
        assert t.dtype == np.uint16 and t.shape == shape, k
    assert inp.shape == (M, N, K)
    assert _std_ok(inp.W, 0.02, inp.W.size)
    assert abs(inp.W.mean()) < 6 * 0.02 / math.sqrt(inp.W.size)
    # bf16 tensors carry the rounding of their fp32 draws: std within sampling error plus 2^-8
    for k, want in (("X", 1.0), ("A", 1.0 / math.sqrt(K)), ("B", 0.01), ("G", 1.0)):
        x = _bf16_to_f64(getattr(inp, k))
        assert abs(np.std(x) / want - 1.0) < 6.0 / math.sqrt(2.0 * x.size) + 2.0 ** -8, k


def test_bf16_bits_are_round_to_nearest_even_of_the_draw():
    g = synth.rng(902, synth.S_X)
    x = synth.normal_f32(g, (4096,), 1.0)
    np.testing.assert_array_equal(synth.to_bf16_bits(x), _bf16_rne(x))
    # ties go to even: 1 + 2^-8 lies halfway between two bf16 neighbours
    ties = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8)], np.float32)
    np.testing.assert_array_equal(synth.to_bf16_bits(ties), _bf16_rne(ties))
    np.testing.assert_array_equal(synth.to_bf16_bits(ties), np.array([0x3F80, 0x3F82, 0xBF80], np.uint16))


@pytest.mark.parametrize("kind", ["uniform", "t3"])
def test_weight_outliers(kind):
    rows, cols, std = 1024, 4096, 0.02
    n = rows * cols
    w = synth.weight(903, rows, cols, std, outliers=kind)
    base = synth.weight(903, rows, cols, std)
    changed = w != base
    k = int(changed.sum())
    # 0.1% of the entries, within 6 binomial standard deviations
    assert abs(k - 0.001 * n) < 6 * math.sqrt(n * 0.001 * 0.999)
    v = w[changed]
    if kind == "uniform":
        assert np.all(np.abs(v) >= 0.2) and np.all(np.abs(v) <= 1.0)
        assert abs((v > 0).mean() - 0.5) < 6 * math.sqrt(0.25 / k)
    else:
        t = v / std
        # Student-t(3): heavy tails (P(|t| > 5) is about 1.5%, against 6e-7 for a normal) and
        # variance 3 (the sample variance converges slowly; the median of |t| is 0.765)
        assert (np.abs(t) > 5).mean() > 0.005
        assert abs(np.median(np.abs(t)) - 0.765) < 0.06


def test_workload_sizes():
    a = synth.LLAMA8B_ATTN
    assert (a["M"], a["N"], a["K"], a["r"], a["alpha"]) == (4096, 4096, 4096, 16, 32.0)
    m = synth.LLAMA8B_MLP
    assert (m["M"], m["r"], m["alpha"]) == (8192, 64, 128.0)
    assert [x[1:] for x in m["mats"]] == [(14336, 4096), (14336, 4096), (4096, 14336)]
    d = synth.LLAMA70B_DECODE
    assert d["Ms"] == [1, 8, 32] and d["w_std"] == 0.015
    assert sorted(x[1:] for x in d["mats"]) == [(8192, 28672), (28672, 8192)]
    s = synth.LLAMA70B_SWEEP
    assert s["layers"] == 80
    # per layer: q, o 8192^2; k, v 1024 x 8192; gate, up, down 8192 <-> 28672
    assert sum(r * c for _, r, c in s["mats"]) == 2 * 8192 ** 2 + 2 * 1024 * 8192 + 3 * 8192 * 28672
    # rank 16 on all seven linears of Llama-3-8B's 32 blocks: 16 * (N + K) per matrix
    assert synth.adapter_param_count() == 32 * 16 * (2 * 8192 + 2 * 5120 + 3 * 18432) == 41_943_040


def test_adamw_inputs():
    n = 200_001
    o = synth.adamw_inputs(904, n)
    for k in ("p", "g", "m", "v"):
        a = getattr(o, k)
        assert a.dtype == np.float32 and a.shape == (n,), k
    assert np.all(o.v >= 0)
    h = n // 2
    assert np.all(np.abs(o.p[:h]) <= 1 / 64)
    assert _std_ok(o.p[h:], 0.01, n - h)
    for a in (o.g, o.v):  # 1% exact zeros
        z = (a == 0).mean()
        assert abs(z - 0.01) < 6 * math.sqrt(0.01 * 0.99 / n)
    assert _std_ok(o.m, 1e-4, n)
