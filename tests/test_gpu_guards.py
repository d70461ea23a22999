"""Guard bytes around every buffer a call writes.

Each output and each workspace sits between two 4 KiB runs of sentinel bytes (0xA5).  A kernel
that writes past either edge of a ragged shape (a token tail, a weight-row tail, a contraction
tail, an odd rank, a scalar tail of a vector loop) changes a sentinel and fails here.  The
guarded calls must also give, bit for bit, what the same calls give into plain buffers: the
parity of those with the oracle is checked by the other GPU tests."""
import numpy as np
import pytest
import torch

import bit_nf4_quantized_36_b300 as q
from bit_nf4_quantized_36_b300 import synth
from gpu_util import dev_bf16

pytestmark = pytest.mark.gpu

GUARD = 4096
FILL = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_nf4_quantized_36_b300 import build
    build.build()
    yield
    q.check_device_error()


class Guarded:
    """A device buffer of `shape` and `dtype` with GUARD sentinel bytes on each side."""

    def __init__(self, shape, dtype):
        esz = torch.empty((), dtype=dtype).element_size()
        self.n = int(np.prod(shape, dtype=np.int64)) * esz
        self.raw = torch.full((2 * GUARD + self.n,), FILL, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + self.n].view(dtype).view(shape)

    def intact(self) -> bool:
        return bool((self.raw[:GUARD] == FILL).all()) and bool((self.raw[GUARD + self.n:] == FILL).all())


def _check(bufs: dict):
    torch.cuda.synchronize()
    q.check_device_error()
    bad = [k for k, g in bufs.items() if not g.intact()]
    assert not bad, f"writes outside the buffer: {bad}"


def _guarded_nf4(rows, cols):
    n = rows * cols
    nb = n // 64
    parts = dict(codes=Guarded((n // 2,), torch.uint8), scale_codes=Guarded((nb,), torch.int8),
                 scale_scales=Guarded(((nb + 255) // 256,), torch.float32),
                 scale_offset=Guarded((1,), torch.float32))
    w = q.NF4Weight(rows, cols, parts["codes"].t, parts["scale_codes"].t, parts["scale_scales"].t,
                    parts["scale_offset"].t)
    return w, parts


@pytest.mark.parametrize("M,N,K,r", [
    (1, 136, 2112, 3),     # one token: the GEMV, ragged rows, odd rank
    (12, 264, 4160, 8),    # the small-M tensor kernel
    (130, 264, 320, 24),   # the fused GEMM with a ragged token tile, K % 128 != 0
    (257, 136, 192, 5),    # one token past a tile, weight rows past a tile, odd rank
    (600, 520, 640, 16),   # two token tiles per unit, ragged rows
])
def test_layer_calls_stay_inside_their_buffers(M, N, K, r):
    inp = synth.layer_inputs(240 + r, M, N, K, r, 2.0 * r, b_std=0.3)
    W = torch.from_numpy(inp.W).cuda()
    X, A, B, G = (dev_bf16(a) for a in (inp.X, inp.A, inp.B, inp.G))

    # quantize into guarded storage with a guarded workspace
    qw, parts = _guarded_nf4(N, K)
    wsq = Guarded((max(q.quantize_workspace_bytes(N, K), 16),), torch.uint8)
    q.nf4_quantize(W, out=qw, workspace=wsq.t)
    _check({**parts, "ws": wsq})
    ref = q.nf4_quantize(W)
    for k in ("codes", "scale_codes", "scale_scales", "scale_offset"):
        assert torch.equal(getattr(qw, k), getattr(ref, k)), k

    # dequantize
    D = Guarded((N, K), torch.bfloat16)
    q.nf4_dequantize(qw, out=D.t)
    _check({"W^": D})
    assert torch.equal(D.t, q.nf4_dequantize(ref))

    # forward
    Y, U = Guarded((M, N), torch.bfloat16), Guarded((M, r), torch.bfloat16)
    wsf = Guarded((max(q.fwd_workspace_bytes(M, N, K, r), 16),), torch.uint8)
    q.qlora_linear_fwd(qw, X, A, B, inp.alpha, Y=Y.t, U_save=U.t, workspace=wsf.t)
    _check({"Y": Y, "U": U, "ws": wsf})
    Y0, U0 = q.qlora_linear_fwd(ref, X, A, B, inp.alpha)
    assert torch.equal(Y.t, Y0) and torch.equal(U.t, U0)

    # backward
    dX, dA, dB = Guarded((M, K), torch.bfloat16), Guarded((r, K), torch.float32), Guarded((N, r), torch.float32)
    wsb = Guarded((max(q.bwd_workspace_bytes(M, N, K, r), 16),), torch.uint8)
    q.qlora_linear_bwd(qw, X, A, B, inp.alpha, G, U.t, dX=dX.t, dA=dA.t, dB=dB.t, workspace=wsb.t)
    _check({"dX": dX, "dA": dA, "dB": dB, "ws": wsb})
    dX0, dA0, dB0 = q.qlora_linear_bwd(ref, X, A, B, inp.alpha, G, U0)
    assert torch.equal(dX.t, dX0) and torch.equal(dA.t, dA0) and torch.equal(dB.t, dB0)

    # merge
    Wm = Guarded((N, K), torch.bfloat16)
    wsm = Guarded((max(q.merge_workspace_bytes(N, K, r), 16),), torch.uint8)
    q.qlora_merge(qw, A, B, inp.alpha, out=Wm.t, workspace=wsm.t)
    _check({"W_m": Wm, "ws": wsm})
    assert torch.equal(Wm.t, q.qlora_merge(ref, A, B, inp.alpha))


@pytest.mark.parametrize("n", [1, 3, 5, 4099])
def test_adamw_stays_inside_its_buffers(n):
    inp = synth.adamw_inputs(241, n)
    bufs = {k: Guarded((n,), torch.float32) for k in ("p", "g", "m", "v")}
    for k in bufs:
        bufs[k].t.copy_(torch.from_numpy(getattr(inp, k)))
    pb = Guarded((n,), torch.bfloat16)
    q.adamw_step(bufs["p"].t, bufs["g"].t, bufs["m"].t, bufs["v"].t, 1, 2e-4, weight_decay=0.01,
                 p_bf16=pb.t)
    _check({**bufs, "p_bf16": pb})
    p, g, m, v = (torch.from_numpy(getattr(inp, k).copy()).cuda() for k in ("p", "g", "m", "v"))
    q.adamw_step(p, g, m, v, 1, 2e-4, weight_decay=0.01)
    assert torch.equal(bufs["p"].t, p) and torch.equal(bufs["m"].t, m) and torch.equal(bufs["v"].t, v)
    assert torch.equal(pb.t, p.to(torch.bfloat16))
