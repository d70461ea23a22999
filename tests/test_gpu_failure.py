"""The device-side failure path, exercised without a fault or a hang.

Every wait of the fused NF4-dequant GEMM on a pipeline barrier is bounded (about 2 s).  The
library's test hook (qlora_test_inject) makes the leader CTA of the first CTA pair leave out the
copy of packed codes for its first k-step, so the barrier its decode warps wait on never
completes: no flag is ever set for them.  The wait runs out, the kernel's roles let their
copies drain and exit, and the host reads QLORA_ERR_TIMEOUT from the device error word.  The
context stays usable: the same calls afterwards give the same bits as before the injection."""
import time

import pytest
import torch

import bit_nf4_quantized_36_b300 as q
from bit_nf4_quantized_36_b300 import _lib, synth
from gpu_util import dev_bf16

pytestmark = pytest.mark.gpu

QLORA_ERR_TIMEOUT = 6


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_nf4_quantized_36_b300 import build
    build.build()
    yield
    q.test_inject(0)


@pytest.mark.parametrize("M,N,K,r", [
    (300, 520, 640, 16),   # one token tile per unit, ragged tokens and weight rows
    (600, 520, 640, 16),   # two token tiles per unit
])
def test_bounded_wait_runs_out_and_the_context_stays_usable(M, N, K, r):
    inp = synth.layer_inputs(230, M, N, K, r, 2.0 * r)
    W = torch.from_numpy(inp.W).cuda()
    X, A, B, G = (dev_bf16(a) for a in (inp.X, inp.A, inp.B, inp.G))
    qw = q.nf4_quantize(W)

    def fwd():
        return q.qlora_linear_fwd(qw, X, A, B, inp.alpha)

    def bwd(U):
        return q.qlora_linear_bwd(qw, X, A, B, inp.alpha, G, U)

    Y0, U0 = fwd()
    dX0, dA0, dB0 = bwd(U0)
    q.check_device_error()

    q.test_inject(_lib.QLORA_INJECT_SKIP_CODES)
    try:
        for call in (fwd, lambda: bwd(U0)):
            t0 = time.monotonic()
            call()
            with pytest.raises(q.QLoRAError) as e:
                q.check_device_error()
            assert e.value.status == QLORA_ERR_TIMEOUT
            assert time.monotonic() - t0 < 30.0
        q.check_device_error()  # read and cleared
    finally:
        q.test_inject(0)

    Y1, U1 = fwd()
    dX1, dA1, dB1 = bwd(U1)
    q.check_device_error()
    for name, a, b in (("Y", Y0, Y1), ("U", U0, U1), ("dX", dX0, dX1), ("dA", dA0, dA1), ("dB", dB0, dB1)):
        assert torch.equal(a, b), name


def test_hook_rejects_unknown_flags():
    with pytest.raises(q.QLoRAError):
        q.test_inject(2)
