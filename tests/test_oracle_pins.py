"""Pins for the CPU oracle: each check ties an oracle routine to something other than itself --
values the pages print (tests/golden/*), closed forms, a library routine for a special case, or
brute force on tiny inputs.  CPU only."""
import math
import statistics
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import golden

F32 = np.float32


# ----------------------------------------------------------------------------------------
# absmax int4 worked example and its error bound
# ----------------------------------------------------------------------------------------

def test_int4_worked_example(orc):
    g = golden("int4_worked_example.txt")
    w = np.array([float(v) for v in g["weights"]], dtype=F32)
    am, codes, w_hat = orc.int4_absmax(w)
    assert am == pytest.approx(float(g["absmax"][0]))
    assert codes.tolist() == [int(v) for v in g["codes"]]
    assert [f"{v:.2f}" for v in w_hat] == [f"{float(v):.2f}" for v in g["restored_2dp"]]
    assert f"{np.abs(w - w_hat).max():.3f}" == g["max_error_3dp"][0]
    assert f"{am / 14:.3f}" == g["bound_3dp"][0]
    w2 = w.copy()
    w2[int(g["outlier_index"][0])] = float(g["outlier_value"][0])
    _, codes2, _ = orc.int4_absmax(w2)
    assert codes2.tolist() == [int(v) for v in g["outlier_codes"]]


def test_int4_error_bound_random_blocks(orc):
    # |w - w^| <= absmax / 14 (half a step); fp32 rounding adds at most a few ulp of absmax
    g = np.random.default_rng(1)
    for _ in range(200):
        w = (g.standard_normal(64) * g.uniform(0.01, 3)).astype(F32)
        am, codes, w_hat = orc.int4_absmax(w)
        assert np.all(np.abs(codes) <= 7)
        assert np.abs(w.astype(np.float64) - w_hat).max() <= am / 14 * (1 + 1e-5)


# ----------------------------------------------------------------------------------------
# Phi^{-1} and the level tables
# ----------------------------------------------------------------------------------------

def test_norm_ppf_matches_library(orc):
    nd = statistics.NormalDist()
    for p in [1e-6, 0.01, 0.03, 0.1, 0.25, 0.4999, 0.5, 0.5001, 0.75, 0.9, 0.9677083, 0.99, 1 - 1e-6]:
        assert orc.norm_ppf(p) == pytest.approx(nd.inv_cdf(p), rel=1e-13, abs=1e-15)
    assert orc.norm_ppf(0.975) == pytest.approx(1.959963984540054, rel=1e-14)


def test_toy_table_matches_printed(orc):
    g = golden("toy_nf4_table.txt")
    toy = orc.toy_levels(float(g["d"][0]))
    assert [f"{v:+.2f}" for v in toy] == g["levels_2dp"]
    # the int4 comparator of the same section: 15 levels, step 1/7
    assert len(np.arange(-7, 8)) == int(g["int4_levels"][0])
    assert f"{round(1 / 7, 3):.3f}" == g["int4_step_3dp"][0]


def _nf4_from_library():
    """NF4 levels of the ultralytics snippet, computed with statistics.NormalDist in fp64."""
    nd = statistics.NormalDist()
    top = 0.9677083
    pos = [nd.inv_cdf(top + (0.5 - top) * i / 8) for i in range(8)]
    neg = [-nd.inv_cdf(top + (0.5 - top) * j / 7) for j in range(7)]
    v = sorted(neg + [0.0] + pos)
    return np.array([x / v[-1] for x in v], dtype=F32)


def test_nf4_levels_structure_and_library(orc):
    L = orc.nf4_levels()
    assert L.dtype == F32 and L.size == 16
    assert L[0] == -1.0 and L[15] == 1.0 and L[7] == 0.0
    assert np.all(np.diff(L) > 0)
    assert (L < 0).sum() == 7 and (L > 0).sum() == 8
    # not mirror-symmetric: 7 negative vs 8 positive quantiles
    assert -L[6] != L[8]
    np.testing.assert_array_equal(L.view(np.uint32), _nf4_from_library().view(np.uint32))
    # each half is +-Phi^{-1} of evenly spaced probabilities
    x_max = statistics.NormalDist().inv_cdf(0.9677083)
    for i, p in enumerate(np.linspace(0.9677083, 0.5, 9)[:-1]):
        assert L[15 - i] == pytest.approx(statistics.NormalDist().inv_cdf(p) / x_max, rel=1e-6)


def test_nf4_vs_uniform_mse_matches_printed(orc):
    g = golden("nf4_vs_uniform_mse.txt")
    torch.manual_seed(int(g["seed"][0]))
    rows, cols = (int(v) for v in g["shape"])
    w = (torch.randn(rows, cols) * float(g["std"][0])).numpy()
    mse_nf4 = orc.blockwise_mse(w, 64, orc.nf4_levels())
    uniform = torch.linspace(-1, 1, 16).numpy()
    mse_uni = orc.blockwise_mse(w, 64, uniform)
    assert f"{mse_nf4:.3e}" == g["nf4_mse_4sig"][0]
    assert f"{mse_uni:.3e}" == g["uniform16_mse_4sig"][0]
    assert abs((1 - mse_nf4 / mse_uni) * 100 - float(g["reduction_percent_approx"][0])) < 1.0


def test_nf4_mse_statistical_other_seeds(orc):
    # same experiment on other draws: the ratio stays in the band the printed values imply
    for seed in range(3):
        w = (np.random.default_rng(100 + seed).standard_normal((4096, 64)) * 0.02).astype(F32)
        a = orc.blockwise_mse(w, 64, orc.nf4_levels())
        b = orc.blockwise_mse(w, 64, np.linspace(-1, 1, 16).astype(F32))
        assert a == pytest.approx(3.395e-06, rel=0.03)
        assert b == pytest.approx(4.053e-06, rel=0.03)
        assert 0.80 < a / b < 0.88


# ----------------------------------------------------------------------------------------
# NF4 codes: brute force, invariants, packing
# ----------------------------------------------------------------------------------------

def _brute_codes(w, L):
    w = np.asarray(w, F32).reshape(-1, 64)
    am = np.abs(w).max(axis=1, keepdims=True)
    out = np.zeros(w.shape, dtype=np.uint8)
    for b in range(w.shape[0]):
        for i in range(64):
            if am[b, 0] == 0:
                out[b, i] = 7
                continue
            x = F32(w[b, i] / am[b, 0])
            d = [abs(F32(x - L[k])) for k in range(16)]
            out[b, i] = d.index(min(d))  # first minimum
    return out.reshape(-1), am.reshape(-1)


def test_nf4_codes_brute_force_tiny(orc):
    L = orc.nf4_levels()
    g = np.random.default_rng(7)
    w = (g.standard_normal(64 * 24) * 0.02).astype(F32)
    w[64:128] = 0.0                       # all-zero block
    w[128:192] = np.abs(w[128:192])       # one-signed block
    codes, am = orc.blockwise_codes(w, 64, L)
    bc, bam = _brute_codes(w, L)
    np.testing.assert_array_equal(codes, bc)
    np.testing.assert_array_equal(am, bam)
    # numpy's argmin (first occurrence) on the fp32 distance matrix, away from all-zero blocks
    x = (w.reshape(-1, 64) / np.where(bam == 0, 1, bam)[:, None]).astype(F32).reshape(-1)
    ref = np.argmin(np.abs(x[:, None] - L[None, :]).astype(F32), axis=1)
    nz = np.repeat(bam != 0, 64)
    np.testing.assert_array_equal(codes[nz], ref[nz])


def test_nf4_codes_ties_go_to_lower_index(orc):
    # x exactly halfway (in fp32) between two levels must take the lower index
    L = orc.nf4_levels()
    hits = 0
    for k in range(15):
        m = F32((np.float64(L[k]) + np.float64(L[k + 1])) / 2)
        for x in (np.nextafter(m, F32(-2)), m, np.nextafter(m, F32(2))):
            d = [abs(F32(F32(x) - L[j])) for j in range(16)]
            want = d.index(min(d))
            blk = np.zeros(64, F32)
            blk[0] = 1.0
            blk[1] = x
            codes, _ = orc.blockwise_codes(blk, 64, L)
            assert codes[1] == want
            if d[k] == d[k + 1]:
                assert want == k
                hits += 1
    assert hits >= 1  # at least one exact fp32 tie is exercised


def test_nf4_codes_invariants(orc):
    L = orc.nf4_levels()
    w = (np.random.default_rng(3).standard_normal(64 * 500) * 0.02).astype(F32)
    codes, am = orc.blockwise_codes(w, 64, L)
    cb = codes.reshape(-1, 64)
    wb = w.reshape(-1, 64)
    arg = np.abs(wb).argmax(axis=1)
    mx_codes = cb[np.arange(cb.shape[0]), arg]
    assert np.all((mx_codes == 0) | (mx_codes == 15))
    # reconstruction error <= half the widest gap (between L0 and L1) times absmax
    half_gap = (L[1] - L[0]) / 2
    err = np.abs(wb - L[cb] * am[:, None])
    assert np.all(err <= half_gap * am[:, None] * (1 + 1e-6))
    # zero weights get the exact-zero level
    z = np.zeros(64, F32)
    z[5] = 0.3
    c, _ = orc.blockwise_codes(z, 64, L)
    assert c[0] == 7 and c[5] == 15


def test_pack_nibbles_order(orc):
    codes = np.array([1, 2, 15, 0, 7, 8], dtype=np.uint8)
    packed = orc.pack_nibbles(codes)
    assert packed.tolist() == [0x12, 0xF0, 0x78]
    np.testing.assert_array_equal(orc.unpack_nibbles(packed), codes)


# ----------------------------------------------------------------------------------------
# Double quantization
# ----------------------------------------------------------------------------------------

def _exact_f32_round(fr: Fraction) -> np.float32:
    """Round an exact rational to the nearest fp32 (ties to even), without double rounding."""
    c = np.float32(float(fr))
    best = None
    for cand in (np.nextafter(c, F32(-np.inf)), c, np.nextafter(c, F32(np.inf))):
        d = abs(Fraction(float(cand)) - fr)
        key = (d, int(np.array(cand, F32).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, cand)
    return F32(best[1])


def test_dq_mean_close_to_exact_mean(orc):
    g = np.random.default_rng(11)
    for nb in (1, 255, 256, 257, 1000, 4096 + 3):
        s = np.abs(g.standard_normal(nb) * 0.05).astype(F32) + F32(0.01)
        mu = orc.dq_mean(s)
        exact = sum(Fraction(float(v)) for v in s) / nb
        ref = _exact_f32_round(exact)
        assert abs(int(np.array(mu).view(np.int32)) - int(np.array(ref).view(np.int32))) <= 1


def test_dq_mean_tree_order_worked_example(orc):
    """The mean's rounding order (reading: in-order fp64 group sums, then a pairwise tree over
    them, elements 2i and 2i + 1 at each level, then one rounding of total / nb to fp32), on four
    groups built so that the order decides the fp32 result.  By hand, with S = (2^53 + 2^29, 1,
    0, 1): S0 + S1 is a tie in fp64 (ulp 2) and stays 2^53 + 2^29; S2 + S3 = 1; their sum is the
    same tie again, so the total is 2^53 + 2^29 and total / 1024 = 2^43 + 2^19, exactly half an
    fp32 ulp above 2^43: ties to even give 2^43.  (Pairing S0 with S2 instead would keep both 1s,
    give 2^43 + 2^19 + 2^-9 and round up to 2^43 + 2^20.)"""
    s = np.zeros(1024, F32)
    s[0], s[1] = 2.0 ** 53, 2.0 ** 29
    s[256] = 1.0
    s[768] = 1.0
    assert float(orc.dq_mean(s)) == 2.0 ** 43


def test_double_quant_invariants(orc):
    g = np.random.default_rng(12)
    s = np.abs(g.standard_normal(256 * 5 + 77) * 0.05).astype(F32) + F32(0.01)
    q, c2, mu = orc.double_quant(s)
    assert q.size == s.size and c2.size == 6
    for gi in range(c2.size):
        seg = s[gi * 256:(gi + 1) * 256]
        d = (seg - mu).astype(F32)
        assert c2[gi] == np.abs(d).max()
        qs = q[gi * 256:(gi + 1) * 256]
        j = int(np.abs(d).argmax())
        assert qs[j] == (127 if d[j] > 0 else -127)
        assert np.all(np.abs(qs.astype(int)) <= 127)
        # sign of the code follows the sign of s - mu (or is zero)
        assert np.all(np.sign(qs) * np.sign(d) >= 0)
        rebuilt = np.array([orc.dq_scale(int(a), float(c2[gi]), float(mu)) for a in qs], dtype=F32)
        ulp = np.spacing(np.maximum(np.abs(seg), np.abs(rebuilt)))
        assert np.all(np.abs(rebuilt.astype(np.float64) - seg) <= c2[gi] / 254.0 + 2 * ulp)


def test_double_quant_degenerate_group(orc):
    s = np.full(300, 0.0625, dtype=F32)  # every scale equal: mu is exact, c2 = 0, q = 0
    q, c2, mu = orc.double_quant(s)
    assert mu == F32(0.0625) and np.all(c2 == 0) and np.all(q == 0)
    assert orc.dq_scale(0, 0.0, float(mu)) == F32(0.0625)


def test_dq_scale_is_single_rounding_fma(orc):
    g = np.random.default_rng(13)
    for _ in range(300):
        q = int(g.integers(-127, 128))
        c2 = F32(abs(g.standard_normal()) * 0.03)
        mu = F32(abs(g.standard_normal()) * 0.05)
        k = F32(c2 / F32(127.0))
        exact = Fraction(q) * Fraction(float(k)) + Fraction(float(mu))
        assert orc.dq_scale(q, float(c2), float(mu)) == _exact_f32_round(exact)


# ----------------------------------------------------------------------------------------
# bf16 rounding and dequantization
# ----------------------------------------------------------------------------------------

def test_bf16_round_matches_torch(orc):
    g = np.random.default_rng(14)
    vals = list((g.standard_normal(3000) * 10.0 ** g.integers(-30, 30, 3000)).astype(F32))
    # exact ties and near-overflow values
    for base in (0x3F808000, 0x3F818000, 0x7F7F8000, 0xFF7F8000, 0x00008000, 0x7F7FFFFF, 0x3F80FFFF):
        vals.append(np.array([base], dtype=np.uint32).view(F32)[0])
    vals += [F32(0.0), F32(-0.0), F32(1.0), F32(np.inf), F32(-np.inf)]
    a = np.array(vals, dtype=F32)
    want = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.bf16_round_array(a)
    np.testing.assert_array_equal(got, want)


def test_bf16_round_keeps_nan_a_nan(orc):
    """NaN inputs (outside the layer's contract, which wants finite weights) must not turn into
    infinities or numbers: whatever the payload, the result has an all-ones exponent and a
    non-zero significand, and keeps its sign."""
    for bits in (0x7F800001, 0x7FC00000, 0x7FA00000, 0x7F80FFFF, 0xFF800001, 0xFFFFFFFF):
        x = np.array([bits], dtype=np.uint32).view(F32)[0]
        h = int(orc.bf16_round(x))
        assert (h & 0x7F80) == 0x7F80 and (h & 0x007F) != 0, hex(bits)
        assert (h >> 15) == (bits >> 31), hex(bits)


def test_dequantize_definition_small(orc):
    W = (np.random.default_rng(15).standard_normal((8, 128)) * 0.02).astype(F32)
    W[2, :64] = 0.0
    qz = orc.nf4_quantize(W)
    Wh = orc.nf4_dequantize(qz["packed"], qz["qcode"], qz["c2"], qz["mu"], 8, 128)
    L = orc.nf4_levels()
    codes = orc.unpack_nibbles(qz["packed"])
    for i in range(W.size):
        b = i // 64
        s = orc.dq_scale(int(qz["qcode"][b]), float(qz["c2"][b // 256]), float(qz["mu"]))
        v = torch.tensor([F32(L[codes[i]] * s)], dtype=torch.float32).to(torch.bfloat16)
        assert int(v.view(torch.int16).numpy().view(np.uint16)[0]) == int(Wh.reshape(-1)[i])
    # the reconstruction stays near W: NF4 half-gap plus the double-quant step of the scale
    Wf = orc.bf16_to_f64(Wh)
    am = qz["absmax"].reshape(8, 2)
    step = qz["c2"][0] / 254.0
    bound = 0.1520 * (np.repeat(am, 64, axis=1) + step) + step + np.abs(W) * 2 ** -8
    assert np.all(np.abs(Wf - W) <= bound + 1e-7)


def test_dequantize_definition_several_groups(orc):
    """The same definition over 512 blocks in two groups of different magnitude, so that each
    block must take its own group's constant c2_g."""
    W = (np.random.default_rng(16).standard_normal((4, 8192)) * 0.02).astype(F32)
    W[2:] *= 50.0                                    # the second group's scales are 50x larger
    qz = orc.nf4_quantize(W)
    # both constants measure from the common mean: they differ, though by less than 50x
    assert qz["c2"].size == 2 and qz["c2"][1] > 1.5 * qz["c2"][0]
    Wh = orc.nf4_dequantize(qz["packed"], qz["qcode"], qz["c2"], qz["mu"], 4, 8192).reshape(-1)
    L = orc.nf4_levels()
    codes = orc.unpack_nibbles(qz["packed"])
    s = np.array([orc.dq_scale(int(qz["qcode"][b]), float(qz["c2"][b // 256]), float(qz["mu"]))
                  for b in range(qz["qcode"].size)], dtype=F32)
    v = (L[codes].astype(F32) * np.repeat(s, 64)).astype(F32)          # one fp32 rounding
    want = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(Wh, want)


def test_storage_bits_closed_form(orc):
    g = golden("storage_bits.txt")
    n = int(g["params"][0])
    n64 = (n // 16384) * 16384  # a matrix size with whole groups
    bits = 8 * orc.nf4_storage_bytes(n64 // 64, 64) / n64
    assert f"{bits:.3f}" == g["bits_double"][0]
    for key, b in (("bits_fp32", 32), ("bits_bf16", 16), ("bits_absmax", 4 + 32 / 64)):
        assert f"{b:.3f}" == g[key][0]
    assert f"{n * 4.5 / 8e9:.2f}" == g["gb_absmax"][0]
    assert f"{n * 32 / 8e9:.2f}" == g["gb_fp32"][0]
    assert f"{n * 16 / 8e9:.2f}" == g["gb_bf16"][0]
    assert f"{orc.nf4_storage_bytes(n64 // 64, 64) / 1e9:.2f}" == g["gb_double"][0]
    n65 = int(g["params_65b"][0])
    gb = orc.nf4_storage_bytes(n65 // 64 // 64 * 64, 64) / 1e9
    assert abs(gb - float(g["gb_65b_approx"][0])) < 1.0


def test_storage_bytes_by_enumeration(orc):
    """Brute force on small matrices, counted item by item as the stored format lists them: a
    4-bit code per weight, an int8 scale code per 64-weight block, an fp32 constant per started
    group of 256 blocks, and the fp32 mean of the scales once per matrix. The shapes include a
    last group that is only partly filled."""
    for rows, cols in [(1, 64), (64, 64), (3, 4096), (257, 128), (1024, 1024)]:
        bits = 0
        blocks = 0
        for w in range(rows * cols):
            bits += 4
            if w % 64 == 63:
                blocks += 1
                bits += 8
                if blocks % 256 == 1:   # the first block of a group opens it
                    bits += 32
        bits += 32                      # the mean
        assert orc.nf4_storage_bytes(rows, cols) * 8 == bits, (rows, cols)
        # and the quantizer's outputs are exactly those items
        q = orc.nf4_quantize(np.zeros((rows, cols), F32))
        stored = q["packed"].nbytes + q["qcode"].nbytes + q["c2"].nbytes + np.float32(q["mu"]).nbytes
        assert stored * 8 == bits, (rows, cols)


# ----------------------------------------------------------------------------------------
# The layer: explicit effective matrix, finite differences, special cases
# ----------------------------------------------------------------------------------------

def _bf16(x):
    return torch.from_numpy(np.asarray(x, F32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _small_layer(seed, M=5, N=6, K=128, r=3, b_std=0.3):
    g = np.random.default_rng(seed)
    What = _bf16(g.standard_normal((N, K)) * 0.05)
    X = _bf16(g.standard_normal((M, K)))
    A = _bf16(g.standard_normal((r, K)) * 0.1)
    B = _bf16(g.standard_normal((N, r)) * b_std)
    G = _bf16(g.standard_normal((M, N)))
    return What, X, A, B, G


def test_layer_against_effective_matrix(orc):
    What, X, A, B, G = _small_layer(21)
    alpha, r = 8.0, A.shape[0]
    s = alpha / r
    f = orc.bf16_to_f64
    Weff = f(What) + s * (f(B) @ f(A))           # (W^ + s B A), the page's gradient formula
    Y, U = orc.layer_fwd_rows(What, X, A, B, alpha)
    np.testing.assert_allclose(Y, f(X) @ Weff.T, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(U, f(X) @ f(A).T, rtol=1e-12, atol=1e-12)
    dX = orc.layer_dx_rows(What, A, B, G, alpha)
    np.testing.assert_allclose(dX, f(G) @ Weff, rtol=1e-12, atol=1e-12)
    rows = np.array([4, 1], dtype=np.int64)
    Ys, _ = orc.layer_fwd_rows(What, X, A, B, alpha, rows)
    np.testing.assert_array_equal(Ys, Y[rows])


def test_layer_grads_finite_differences(orc):
    What, X, A, B, G = _small_layer(22, M=4, N=5, K=64, r=2)
    alpha = 4.0
    f = orc.bf16_to_f64
    s = alpha / A.shape[0]

    def loss(Xf, Af, Bf):
        return float(np.sum(f(G) * (Xf @ f(What).T + s * (Xf @ Af.T) @ Bf.T)))

    dA, dB = orc.layer_adapter_grads(X, A, B, G, alpha)
    dX = orc.layer_dx_rows(What, A, B, G, alpha)
    Xf, Af, Bf = f(X), f(A), f(B)
    h = 1e-3
    for (j, k) in [(0, 0), (1, 17), (0, 63)]:
        E = np.zeros_like(Af)
        E[j, k] = h
        fd = (loss(Xf, Af + E, Bf) - loss(Xf, Af - E, Bf)) / (2 * h)
        assert dA[j, k] == pytest.approx(fd, rel=1e-7, abs=1e-9)
    for (n, j) in [(0, 0), (4, 1), (2, 1)]:
        E = np.zeros_like(Bf)
        E[n, j] = h
        fd = (loss(Xf, Af, Bf + E) - loss(Xf, Af, Bf - E)) / (2 * h)
        assert dB[n, j] == pytest.approx(fd, rel=1e-7, abs=1e-9)
    for (m, k) in [(0, 0), (3, 40)]:
        E = np.zeros_like(Xf)
        E[m, k] = h
        fd = (loss(Xf + E, Af, Bf) - loss(Xf - E, Af, Bf)) / (2 * h)
        assert dX[m, k] == pytest.approx(fd, rel=1e-7, abs=1e-9)


def test_layer_special_cases(orc):
    What, X, A, B, G = _small_layer(23)
    alpha = 6.0
    f = orc.bf16_to_f64
    Bz = np.zeros_like(B)
    Y, U = orc.layer_fwd_rows(What, X, A, Bz, alpha)
    np.testing.assert_allclose(Y, f(X) @ f(What).T, rtol=1e-13)
    dA, dB = orc.layer_adapter_grads(X, A, Bz, G, alpha)
    assert np.all(dA == 0)
    np.testing.assert_allclose(dB, alpha / A.shape[0] * f(G).T @ U, rtol=1e-12)
    Wz = np.zeros_like(What)
    Y2, U2 = orc.layer_fwd_rows(Wz, X, A, B, alpha)
    np.testing.assert_allclose(Y2, alpha / A.shape[0] * U2 @ f(B).T, rtol=1e-12)


def test_sampled_adapter_grads_match_full(orc):
    What, X, A, B, G = _small_layer(24, M=7, N=9, K=64, r=4)
    dA, dB = orc.layer_adapter_grads(X, A, B, G, 3.0)
    js = np.array([3, 0], dtype=np.int64)
    dAs, dBt = orc.layer_adapter_grads_cols(X, A, B, G, 3.0, js)
    np.testing.assert_allclose(dAs, dA[js], rtol=1e-13)
    np.testing.assert_allclose(dBt, dB[:, js].T, rtol=1e-13)


# ---------------------------------------------------------------------------------------
# Adapter merge: "QLoRA" (ultralytics), "Compromissos": to merge the adapters the base weight is
# first dequantized to 16 bits; W_m = bf16(W^ + (alpha/r) B A), rounded once.
# ---------------------------------------------------------------------------------------

def _bf16_of_fraction(x):
    """Round an exact rational to bf16 (nearest, ties to even), independently of the oracle:
    exact rational arithmetic on the two 8-bit-significand neighbours."""
    from fractions import Fraction
    x = Fraction(x)
    if x == 0:
        return 0
    sign = 0x8000 if x < 0 else 0
    a = abs(x)
    e = 0
    while a >= 2 ** (e + 1):
        e += 1
    while a < Fraction(2) ** e:
        e -= 1
    step = Fraction(2) ** (e - 7)          # 8 significant bits in [2^e, 2^(e+1))
    m = a // step                          # integer in [128, 256)
    lo, hi = m * step, (m + 1) * step
    if a - lo < hi - a or (a - lo == hi - a and m % 2 == 0):
        v = lo
    else:
        v = hi
    bits = np.array([float(v)], dtype=np.float32).view(np.uint32)[0]
    return sign | int(bits >> 16)


def test_bf16_round_d_agrees_with_fp32_rounding(orc):
    rng = np.random.default_rng(7)
    xs = np.concatenate([rng.standard_normal(3000).astype(np.float32) * 0.02,
                         rng.standard_normal(1000).astype(np.float32) * 1e30,
                         (rng.standard_normal(500) * 1e-39).astype(np.float32),
                         np.array([1.0, -1.0, 3.0e38, 1.00390625, 1.01171875], dtype=np.float32)])
    for x in xs:
        assert orc.bf16_round_d(float(x)) == orc.bf16_round(float(x))


def test_bf16_round_d_rounds_once(orc):
    # 1 + 2^-8 + 2^-30: fp32 would round it to the tie 1 + 2^-8 (then bf16 -> 1.0); one rounding
    # from the exact value gives 1 + 2^-7.
    assert orc.bf16_round_d(1.0 + 2.0 ** -8 + 2.0 ** -30) == 0x3F81
    assert orc.bf16_round_d(1.0 + 2.0 ** -8) == 0x3F80           # tie -> even significand
    assert orc.bf16_round_d(1.0 + 3 * 2.0 ** -8) == 0x3F82       # tie -> even significand


def test_merge_with_zero_adapter_is_the_dequantized_weight(orc):
    rng = np.random.default_rng(11)
    W = (rng.standard_normal((8, 128)) * 0.02).astype(np.float32)
    q = orc.nf4_quantize(W)
    What = orc.nf4_dequantize(q["packed"], q["qcode"], q["c2"], q["mu"], 8, 128)
    A = orc.bf16_round_array(rng.standard_normal((4, 128)).astype(np.float32))
    B = np.zeros((8, 4), dtype=np.uint16)
    assert np.array_equal(orc.merge(What, A, B, 8.0), What)


def test_merge_closed_form(orc):
    from fractions import Fraction
    rng = np.random.default_rng(12)
    W = (rng.standard_normal((6, 64)) * 0.5).astype(np.float32)
    q = orc.nf4_quantize(W)
    What = orc.nf4_dequantize(q["packed"], q["qcode"], q["c2"], q["mu"], 6, 64)
    r = 4
    A = np.full((r, 64), 0x3F80, dtype=np.uint16)                                  # 1.0
    B = np.array([[orc.bf16_round(2.0 ** -(j + 4)) for j in range(r)]] * 6, dtype=np.uint16)
    for alpha, delta in ((4.0, Fraction(15, 128)), (8.0, Fraction(15, 64))):     # s = 1, 2
        got = orc.merge(What, A, B, alpha)
        for n in range(6):
            for k in range(64):
                w = Fraction(float(orc.bf16_to_f64(What[n, k:k + 1])[0]))
                assert got[n, k] == _bf16_of_fraction(w + delta)


def test_merge_general_adapters_exact(orc):
    """Non-uniform A and B (small multiples of powers of two, so B A is exact in fp64): every
    element against W^ + s (B A)[n, k] summed in exact rationals over the rank and rounded once."""
    from fractions import Fraction
    rng = np.random.default_rng(13)
    N, K, r, alpha = 5, 64, 3, 6.0                                   # s = 2
    W = (rng.standard_normal((N, K)) * 0.05).astype(np.float32)
    q = orc.nf4_quantize(W)
    What = orc.nf4_dequantize(q["packed"], q["qcode"], q["c2"], q["mu"], N, K)
    Av = rng.integers(-4, 5, size=(r, K)) * 2.0 ** -5
    Bv = rng.integers(-4, 5, size=(N, r)) * 2.0 ** -7
    A = np.array([[orc.bf16_round(x) for x in row] for row in Av], dtype=np.uint16)
    B = np.array([[orc.bf16_round(x) for x in row] for row in Bv], dtype=np.uint16)
    got = orc.merge(What, A, B, alpha)
    s = Fraction(alpha) / r
    for n in range(N):
        for k in range(K):
            w = Fraction(float(orc.bf16_to_f64(What[n, k:k + 1])[0]))
            ba = sum(Fraction(Bv[n, j]) * Fraction(Av[j, k]) for j in range(r))
            assert got[n, k] == _bf16_of_fraction(w + s * ba), (n, k)


def test_merge_ties_round_to_even(orc):
    What = np.full((1, 64), 0x3F80, dtype=np.uint16)                     # 1.0
    A = np.full((1, 64), 0x3F80, dtype=np.uint16)
    B1 = np.array([[orc.bf16_round(2.0 ** -8)]], dtype=np.uint16)         # s B A = 2^-8: a tie
    assert np.all(orc.merge(What, A, B1, 1.0) == 0x3F80)
    B3 = np.array([[orc.bf16_round(3 * 2.0 ** -8)]], dtype=np.uint16)     # 1 + 3 2^-8: a tie
    assert np.all(orc.merge(What, A, B3, 1.0) == 0x3F82)


def test_merge_rounds_once_from_the_exact_sum(orc):
    """W^ + s B A just above a bf16 midpoint by less than half an fp32 ulp: rounded once (the
    reading) it goes up; rounded through fp32 first it would land on the midpoint and go to
    even.  Both signs, and in another binade."""
    A = np.full((2, 64), 0x3F80, dtype=np.uint16)                            # 1.0
    for w_bits, sign in ((0x3F80, 1.0), (0xBF80, -1.0), (0x4100, 1.0)):      # 1, -1, 8
        w = float(orc.bf16_to_f64(np.array([w_bits], np.uint16))[0])
        half_ulp = abs(w) * 2.0 ** -8                                         # bf16 midpoint offset
        B = np.array([[orc.bf16_round(sign * half_ulp), orc.bf16_round(sign * abs(w) * 2.0 ** -30)]] * 1,
                     dtype=np.uint16)
        What = np.full((1, 64), w_bits, dtype=np.uint16)
        got = orc.merge(What, A, B, 2.0)                                      # s = 1
        away = w_bits + 1                                                     # the next bf16 magnitude
        assert np.all(got == away), (hex(w_bits), hex(int(got[0, 0])))


# ---------------------------------------------------------------------------------------
# LoRA dropout on the adapter input ("LoRA y QLoRA ...", coddykit, LoraConfig lora_dropout=0.05).
# The mask generator is Philox4x32-10 (Salmon et al., "Parallel random numbers: as easy as 1, 2,
# 3", SC'11); its published known-answer vectors pin the oracle's implementation.
# ---------------------------------------------------------------------------------------

def test_philox_known_answer_vectors(orc):
    assert list(orc.philox4x32_10([0, 0, 0, 0], [0, 0])) == [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]
    assert list(orc.philox4x32_10([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2)) == [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]
    assert list(orc.philox4x32_10([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0])) == \
        [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]


def test_dropout_mask_rate_and_layout(orc):
    p = 0.05
    D = orc.dropout_scale(1234, 0, p, 400, 512)
    keep = D != 0
    n = keep.size
    assert np.all(D[keep] == 1.0 / (1.0 - p))
    frac = keep.mean()
    assert abs(frac - (1 - p)) < 5 * np.sqrt(p * (1 - p) / n)
    # element e uses word e % 4 of block e // 4: the kept flags follow the generator directly
    thr = int(np.floor(p * 2.0 ** 32))
    for e in (0, 1, 2, 3, 4, 77, n - 1):
        w = orc.philox4x32_10([e // 4, 0, 0, 0], [1234, 0])[e % 4]
        assert keep.flat[e] == (int(w) >= thr)
    # the full layout at p = 0.5 (every flag a coin toss, so a wrong word, counter or key shows):
    # counter (e / 4 low, e / 4 high, offset low, offset high), key (seed low, seed high)
    seed, offset = (7 << 32) | 0x1234, (5 << 32) | 3
    Dh = orc.dropout_scale(seed, offset, 0.5, 8, 128)
    for e in range(Dh.size):
        w = orc.philox4x32_10([e // 4, 0, offset & 0xFFFFFFFF, offset >> 32], [seed & 0xFFFFFFFF, seed >> 32])[e % 4]
        assert (Dh.flat[e] != 0) == (int(w) >= 2 ** 31), e
    # a different offset gives a different mask; p = 0.5: neighbouring flags look independent
    assert not np.array_equal(keep, orc.dropout_scale(1234, 1, p, 400, 512) != 0)
    k2 = orc.dropout_scale(99, 7, 0.5, 400, 512) != 0
    both = (k2.flat[:-1] & k2.flat[1:]).mean()
    assert abs(both - 0.25) < 5 * np.sqrt(0.25 * 0.75 / (k2.size - 1))


def test_dropout_p0_is_the_plain_layer(orc):
    What, X, A, B, G = _small_layer(24, M=5, N=6, K=64, r=3)
    alpha = 6.0
    D = orc.dropout_scale(5, 0, 0.0, 5, 64)
    assert np.all(D == 1.0)
    Y0, U0 = orc.layer_fwd_rows(What, X, A, B, alpha)
    Y1, U1 = orc.layer_fwd_rows_drop(What, X, A, B, alpha, D)
    assert np.array_equal(Y0, Y1) and np.array_equal(U0, U1)
    assert np.array_equal(orc.layer_dx_rows(What, A, B, G, alpha), orc.layer_dx_rows_drop(What, A, B, G, alpha, D))
    for a, b in zip(orc.layer_adapter_grads(X, A, B, G, alpha), orc.layer_adapter_grads_drop(X, A, B, G, alpha, D)):
        assert np.array_equal(a, b)


def test_dropout_grads_finite_differences(orc):
    What, X, A, B, G = _small_layer(25, M=4, N=5, K=64, r=2)
    alpha = 4.0
    f = orc.bf16_to_f64
    s = alpha / A.shape[0]
    D = orc.dropout_scale(77, 3, 0.3, 4, 64)
    assert (D == 0).any() and (D != 0).any()

    def loss(Xf, Af, Bf):
        return float(np.sum(f(G) * (Xf @ f(What).T + s * ((Xf * D) @ Af.T) @ Bf.T)))

    dA, dB = orc.layer_adapter_grads_drop(X, A, B, G, alpha, D)
    dX = orc.layer_dx_rows_drop(What, A, B, G, alpha, D)
    Xf, Af, Bf = f(X), f(A), f(B)
    # the oracle's forward is the expression differentiated here (the mask on the adapter input
    # only), evaluated with the adapters merged first: X W^T + s (X o D) (B A)^T
    Yd, _ = orc.layer_fwd_rows_drop(What, X, A, B, alpha, D)
    np.testing.assert_allclose(Yd, Xf @ f(What).T + s * (Xf * D) @ (Bf @ Af).T, rtol=1e-12, atol=1e-12)
    h = 1e-3
    for (j, k) in [(0, 0), (1, 17), (0, 63)]:
        E = np.zeros_like(Af)
        E[j, k] = h
        assert dA[j, k] == pytest.approx((loss(Xf, Af + E, Bf) - loss(Xf, Af - E, Bf)) / (2 * h), rel=1e-7, abs=1e-9)
    for (n, j) in [(0, 0), (4, 1), (2, 1)]:
        E = np.zeros_like(Bf)
        E[n, j] = h
        assert dB[n, j] == pytest.approx((loss(Xf, Af, Bf + E) - loss(Xf, Af, Bf - E)) / (2 * h), rel=1e-7, abs=1e-9)
    dropped = np.argwhere(D == 0)[0]
    for (m, k) in [(0, 0), (3, 40), tuple(dropped)]:
        E = np.zeros_like(Xf)
        E[m, k] = h
        assert dX[m, k] == pytest.approx((loss(Xf + E, Af, Bf) - loss(Xf - E, Af, Bf)) / (2 * h), rel=1e-7, abs=1e-9)


# ---------------------------------------------------------------------------------------
# The adapters' optimizer step (AdamW; paged optimizer states, "Otimizadores paginados").
# ---------------------------------------------------------------------------------------

def test_adamw_matches_torch_adamw(orc):
    """torch.optim.AdamW (an independent implementation), in fp64, over 5 steps."""
    rng = np.random.default_rng(31)
    n = 257
    p0 = rng.standard_normal(n)
    grads = [rng.standard_normal(n) * 0.1 for _ in range(5)]
    hp = dict(lr=2e-4, b1=0.9, b2=0.999, eps=1e-8, wd=0.01)
    tp = torch.nn.Parameter(torch.tensor(p0, dtype=torch.float64))
    opt = torch.optim.AdamW([tp], lr=hp["lr"], betas=(hp["b1"], hp["b2"]), eps=hp["eps"], weight_decay=hp["wd"])
    p, m, v = p0.copy(), np.zeros(n), np.zeros(n)
    for t, g in enumerate(grads, start=1):
        tp.grad = torch.tensor(g, dtype=torch.float64)
        opt.step()
        p, m, v = orc.adamw_step(p, g, m, v, hp["lr"], hp["b1"], hp["b2"], hp["eps"], hp["wd"], t)
        np.testing.assert_allclose(p, tp.detach().numpy(), rtol=1e-14, atol=1e-16)


def test_adamw_first_step_is_a_sign_step(orc):
    """t = 1 from zero moments: m^ = g, v^ = g^2, so the step is lr g / (|g| + eps)."""
    g = np.array([0.5, -2.0, 1e-3, -7.0])
    p0 = np.array([1.0, -1.0, 0.25, 3.0])
    lr, wd, eps = 1e-2, 0.1, 1e-8
    p, m, v = orc.adamw_step(p0, g, np.zeros(4), np.zeros(4), lr, 0.9, 0.999, eps, wd, 1)
    np.testing.assert_allclose(p, p0 * (1 - lr * wd) - lr * g / (np.abs(g) + eps), rtol=1e-12)
    np.testing.assert_allclose(m, 0.1 * g, rtol=1e-15)
    np.testing.assert_allclose(v, 0.001 * g * g, rtol=1e-12)
