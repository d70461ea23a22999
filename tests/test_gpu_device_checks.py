"""The device-check build (libqlora_checked.so: the same sources compiled with
QLORA_DEVICE_CHECKS, whose kernels test their global-memory indexes and, on a failed test, latch an
error bit and skip the access instead of trapping).

In a child process that loads the checked library: quantize / dequantize, the layer forward and
backward on each kernel family (the small-M GEMV, the small-M tensor kernel, the CTA-pair kernel
with one and with two token tiles per unit) and the adapter merge, on ragged shapes, must report no
failed check and still match the oracle; then the test hook moves one store index of
nf4_dequantize past the end of its output, and the check must catch it (QLORA_ERR_DEVICE_CHECK,
the store skipped), after which the same call is clean again.  The released library refuses that
hook.  Nothing is written out of bounds in either library."""
import os
import subprocess
import sys

import pytest
import torch

import bit_nf4_quantized_36_b300 as q
from bit_nf4_quantized_36_b300 import _lib

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CHILD = r'''
import sys
sys.path.insert(0, {tests!r})
sys.path.insert(0, {root!r})
import numpy as np
import torch
import oracle
import bit_nf4_quantized_36_b300 as q
from bit_nf4_quantized_36_b300 import _lib, synth
from gpu_util import host_bits, quantize_on_gpu, nf4_to_host, assert_nf4_equal
import test_gpu_layer as tl

assert _lib.LIB_PATH.endswith("libqlora_checked.so"), _lib.LIB_PATH
L = _lib.load()
oracle.lib()
# quantize / dequantize on ragged shapes
for rows, cols in ((1, 64), (72, 192), (300, 320), (129, 1088)):
    W = (np.random.default_rng(rows + cols).standard_normal((rows, cols)) * 0.02).astype(np.float32)
    qw = quantize_on_gpu(W)
    ref = oracle.nf4_quantize(W)
    assert_nf4_equal(nf4_to_host(qw), ref)
    Wh = host_bits(q.nf4_dequantize(qw))
    np.testing.assert_array_equal(Wh, oracle.nf4_dequantize(ref["packed"], ref["qcode"], ref["c2"], ref["mu"], rows, cols))
    q.check_device_error()
# the layer on every kernel family
for M, N, K, r in ((3, 72, 9216, 8), (20, 264, 640, 16), (100, 520, 640, 16), (600, 520, 640, 16)):
    inp = synth.layer_inputs(300 + M, M, N, K, r, 2.0 * r, b_std=0.3)
    tl.check_full(oracle, inp, tl.run_layer(inp))
# the merge
W = torch.randn((264, 576), device="cuda") * 0.02
qw = q.nf4_quantize(W)
A = (torch.randn((16, 576), device="cuda") / 24).to(torch.bfloat16)
B = (torch.randn((264, 16), device="cuda") * 0.01).to(torch.bfloat16)
Wm = q.qlora_merge(qw, A, B, 32.0)
torch.cuda.synchronize()
q.check_device_error()
# the hook: one store index of nf4_dequantize past the end, caught by its check
W = torch.randn((64, 256), device="cuda") * 0.02
qw = q.nf4_quantize(W)
clean = q.nf4_dequantize(qw)
torch.cuda.synchronize()
q.check_device_error()
assert L.qlora_test_inject(_lib.QLORA_INJECT_BOUNDS) == 0
q.nf4_dequantize(qw)
torch.cuda.synchronize()
assert L.qlora_test_inject(0) == 0
try:
    q.check_device_error()
    raise SystemExit("the injected out-of-range index was not reported")
except q.QLoRAError as e:
    assert e.status == 7, e.status  # QLORA_ERR_DEVICE_CHECK
again = q.nf4_dequantize(qw)
torch.cuda.synchronize()
q.check_device_error()
assert torch.equal(again, clean)
print("device checks ok")
'''


@pytest.fixture(scope="module")
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_nf4_quantized_36_b300 import build
    build.build()
    build.build(checks=True)


def test_checked_build_is_clean_and_catches_a_planted_index(_gpu):
    env = dict(os.environ, QLORA_LIB="checked")
    r = subprocess.run([sys.executable, "-c", CHILD.format(tests=HERE, root=ROOT)], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert "device checks ok" in r.stdout


def test_released_library_refuses_the_bounds_hook(_gpu):
    L = _lib.load()
    assert not _lib.LIB_PATH.endswith("libqlora_checked.so")
    assert L.qlora_test_inject(_lib.QLORA_INJECT_BOUNDS) == 1  # QLORA_ERR_INVALID_ARG
    assert L.qlora_test_inject(0) == 0
    q.check_device_error()
