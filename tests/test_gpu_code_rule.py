"""The NF4 code rule (nearest level to x = fl32(w / s_b), ties to the lower level index; "QLoRA"
glossary, ultralytics, NF4 snippet: argmin over |w / absmax - level|) on the GPU against the
oracle, where a division-free shortcut could differ from the rule:

* blocks whose absmax s_b is not a power of two (so fl(w * fl(1/s_b)) need not equal fl(w / s_b)),
  at ordinary, tiny (around 2^-100, where the kernel switches to the exact division), huge (up to
  just below the largest fp32) and subnormal scales, with weights placed so that w / s_b falls
  within 64 ulps of every one of the 15 midpoints between adjacent levels (which also covers
  the exact-tie points next to them);
* every fp32 value x in [-1, 1] (2,130,706,434 values, both zeros included), in blocks whose
  absmax is exactly 1.0, so that x = w, chunked.

Codes are compared bit for bit with the oracle's."""
from concurrent.futures import ThreadPoolExecutor
import os

import numpy as np
import pytest
import torch

import bit_nf4_quantized_36_b300 as q

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_nf4_quantized_36_b300 import build
    build.build()
    yield
    q.check_device_error()


def _threads():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_codes(orc, W2d: np.ndarray) -> np.ndarray:
    """The oracle's packed codes of W2d, its rows split over the host threads (a block's codes
    depend on that block alone, so the split does not change them)."""
    rows = W2d.shape[0]
    T = min(_threads(), max(1, rows // 64))
    cut = [rows * i // T for i in range(T + 1)]
    with ThreadPoolExecutor(T) as ex:
        parts = list(ex.map(lambda i: orc.nf4_quantize(W2d[cut[i]:cut[i + 1]])["packed"], range(T)))
    return np.concatenate(parts)


def _gpu_codes(W2d: np.ndarray) -> np.ndarray:
    qw = q.nf4_quantize(torch.from_numpy(W2d).cuda())
    return qw.codes.cpu().numpy()


def _midpoints(orc):
    L = orc.nf4_levels().astype(np.float64)
    return [np.float32((L[k] + L[k + 1]) / 2) for k in range(15)]


def _scales():
    mant = [1.0, 1.1, 4.0 / 3.0, 1.5, 1.7320508, 1.9999999]
    exps = [-140, -101, -100, -20, 0, 30, 120, 126, 127]
    out = []
    for e in exps:
        for m in mant:
            s = np.float32(m) * np.float32(2.0) ** e if e > -127 else np.float32(m * 2.0 ** e)
            if np.isfinite(s) and s > 0:
                out.append(np.float32(s))
    out.append(np.float32(0.9 * 2.0 ** -100))   # just below the exact-division switch
    out.append(np.float32(3.4e38))              # next to the largest fp32
    return out


def test_code_rule_non_power_of_two_scales_near_thresholds(orc):
    blocks = []
    for s in _scales():
        xs = []
        for c in _midpoints(orc):
            cb = int(np.array([c], np.float32).view(np.int32)[0])
            # 64 fp32 neighbours on each side of the midpoint (the bit patterns of negative
            # values run the other way, which covers the same set)
            xs.append(np.arange(cb - 64, cb + 65, dtype=np.int64).astype(np.uint32).view(np.float32))
        x = np.concatenate(xs)
        w = (x * s).astype(np.float32)  # one fp32 rounding: w / s lands within an ulp or two of x
        w = w[np.isfinite(w) & (np.abs(w) <= s)]
        nb = (w.size + 62) // 63
        pad = np.zeros(nb * 63, np.float32)
        pad[:w.size] = w
        blk = np.concatenate([np.full((nb, 1), s, np.float32), pad.reshape(nb, 63)], axis=1)
        blk[1::2, 0] = -s  # the absmax weight negative in every other block
        blocks.append(blk)
    B = np.concatenate(blocks)
    nb = B.shape[0]
    rows = (nb + 7) // 8 * 8
    Wm = np.zeros((rows, 64), np.float32)
    Wm[:nb] = B
    W2d = Wm.reshape(-1, 512)
    np.testing.assert_array_equal(_gpu_codes(W2d), _oracle_codes(orc, W2d))


def test_code_rule_every_fp32_in_the_unit_interval(orc):
    P = 0x3F800000 + 1                      # +0.0 .. 1.0
    total = 2 * P                           # and -0.0 .. -1.0
    per_chunk = 63 * (1 << 21)              # 2^21 blocks of 63 values + one 1.0 each
    for start in range(0, total, per_chunk):
        i = np.arange(start, min(total, start + per_chunk), dtype=np.int64)
        bits = np.where(i < P, i, 0x80000000 + (i - P)).astype(np.uint32)
        v = bits.view(np.float32)
        nb = (v.size + 62) // 63
        rows = (nb + 63) // 64 * 64
        Wm = np.zeros((rows, 64), np.float32)
        Wm[:, 0] = 1.0
        flat = np.zeros(nb * 63, np.float32)
        flat[:v.size] = v
        Wm[:nb, 1:] = flat.reshape(nb, 63)
        W2d = Wm.reshape(-1, 4096)
        got, want = _gpu_codes(W2d), _oracle_codes(orc, W2d)
        if not np.array_equal(got, want):
            bad = np.nonzero(got != want)[0][:8]
            raise AssertionError(f"codes differ in chunk at {start}: bytes {bad.tolist()}, "
                                 f"gpu {got[bad].tolist()} oracle {want[bad].tolist()}")
