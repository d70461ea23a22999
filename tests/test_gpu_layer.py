"""GPU parity of qlora_linear_fwd / qlora_linear_bwd (through the C ABI) with the fp64 CPU oracle.

The oracle multiplies the bit-exact dequantized bf16 weights in fp64; the GPU accumulates in
fp32 and rounds the LoRA intermediates U, V and the outputs Y, dX to bf16.  Acceptance: relative
Frobenius error <= 5e-3 and max-abs error <= 2e-2 * max|ref| on every compared output."""
import numpy as np
import pytest
import torch

import bit_nf4_quantized_36_b300 as q
from bit_nf4_quantized_36_b300 import synth
from gpu_util import assert_close, dev_bf16, host_bits, host_f64, nf4_to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_nf4_quantized_36_b300 import build
    build.build()
    yield
    q.check_device_error()


def run_layer(inp, fwd_only=False, use_saved_u=True):
    W = torch.from_numpy(inp.W).cuda()
    X, A, B = dev_bf16(inp.X), dev_bf16(inp.A), dev_bf16(inp.B)
    qw = q.nf4_quantize(W)
    Y, U = q.qlora_linear_fwd(qw, X, A, B, inp.alpha)
    out = dict(qw=qw, Y=Y, U=U)
    if not fwd_only:
        G = dev_bf16(inp.G)
        dX, dA, dB = q.qlora_linear_bwd(qw, X, A, B, inp.alpha, G, U if use_saved_u else None)
        out.update(dX=dX, dA=dA, dB=dB)
    torch.cuda.synchronize()
    q.check_device_error()
    return out


_WHAT_CACHE = {}


def oracle_what(orc, inp, qw):
    key = (inp.meta.get("workload"), inp.meta.get("sub"), inp.W.shape, inp.W[:2, :8].tobytes(), inp.W[-1, -8:].tobytes())
    if key not in _WHAT_CACHE:
        ref = orc.nf4_quantize(inp.W)
        N, K = inp.W.shape
        if len(_WHAT_CACHE) >= 2:
            _WHAT_CACHE.pop(next(iter(_WHAT_CACHE)))
        _WHAT_CACHE[key] = (ref["packed"], orc.nf4_dequantize(ref["packed"], ref["qcode"], ref["c2"], ref["mu"], N, K))
    packed, What = _WHAT_CACHE[key]
    np.testing.assert_array_equal(nf4_to_host(qw)["packed"], packed)
    return What


def check_full(orc, inp, out, rows=None, jsel=None):
    What = oracle_what(orc, inp, out["qw"])
    M = inp.X.shape[0]
    sel = np.arange(M) if rows is None else np.asarray(rows)
    Yr, Ur = orc.layer_fwd_rows(What, inp.X, inp.A, inp.B, inp.alpha, sel)
    s = inp.alpha / inp.r
    assert_close("Y", host_f64(out["Y"])[sel], Yr)
    assert_close("U", host_f64(out["U"])[sel], s * Ur)
    if "dX" in out:
        dXr = orc.layer_dx_rows(What, inp.A, inp.B, inp.G, inp.alpha, sel)
        assert_close("dX", host_f64(out["dX"])[sel], dXr)
        if jsel is None:
            dAr, dBr = orc.layer_adapter_grads(inp.X, inp.A, inp.B, inp.G, inp.alpha)
            assert_close("dA", out["dA"].cpu().numpy(), dAr)
            assert_close("dB", out["dB"].cpu().numpy(), dBr)
        else:
            js = np.asarray(jsel)
            dAr, dBt = orc.layer_adapter_grads_cols(inp.X, inp.A, inp.B, inp.G, inp.alpha, js)
            assert_close("dA[j]", out["dA"].cpu().numpy()[js], dAr)
            assert_close("dB[:, j]", out["dB"].cpu().numpy()[:, js].T, dBt)


def test_tiny_workload(orc):
    inp = synth.tiny_inputs()
    check_full(orc, inp, run_layer(inp))


@pytest.mark.parametrize("M,N,K,r", [
    (1, 8, 64, 1),         # smallest everything
    (17, 136, 192, 5),     # ragged tokens, N not a multiple of 128, odd rank
    (130, 264, 320, 24),   # two token tiles with a ragged tail, K % 128 != 0
    (300, 128, 128, 72),   # r64 = 128 (two LoRA k-steps)
    (40, 256, 512, 256),   # maximum rank
    (257, 520, 640, 16),   # token tile 256 + 1, weight tiles 4 + ragged
    (2, 264, 4160, 16),    # two tokens: contraction of 2 full 2048-slices and a 64-wide tail
    (1, 136, 2112, 3),     # one token, odd rank, ragged rows
    (7, 264, 4160, 16),    # seven tokens: eight token columns of the GEMV, one unused
    (8, 136, 2112, 3),     # eight tokens, ragged rows, a contraction tail inside a 256-step
    (3, 72, 9216, 8),      # a row's five 2048-column slabs in two work items (partials added in order)
    (5, 256, 2048, 256),   # the GEMV at the maximum rank: eight adapter row groups, sixteen rank chunks
    (4, 136, 1024, 72),    # the GEMV with a rank that is not a multiple of 32
    (1, 64, 8256, 8),      # the same with a 64-column tail unit (per-unit boxes for the last slab)
    (12, 264, 4160, 8),    # twelve tokens: the small-M tensor kernel
    (600, 520, 640, 16),   # two 256-token tiles per unit: token ranges that cross weight tiles
    (1100, 776, 384, 8),   # the same with more pairs, ragged tokens and weight rows
])
def test_shapes(orc, M, N, K, r):
    inp = synth.layer_inputs(100 + r, M, N, K, r, 2.0 * r, b_std=0.3)
    check_full(orc, inp, run_layer(inp))


def test_saved_u_equals_recomputed_u():
    inp = synth.layer_inputs(201, 96, 256, 384, 16, 32.0)
    a = run_layer(inp, use_saved_u=True)
    b = run_layer(inp, use_saved_u=False)
    for k in ("dX", "dA", "dB"):
        assert torch.equal(a[k], b[k]), k


def test_deterministic():
    inp = synth.layer_inputs(202, 200, 512, 512, 16, 32.0)
    a = run_layer(inp)
    b = run_layer(inp)
    for k in ("Y", "U", "dX", "dA", "dB"):
        assert torch.equal(a[k], b[k]), k


def test_gemv_deterministic():
    """The one-launch GEMV takes its work items from a launch-wide counter (which CTA does which
    item changes from call to call) and still adds every row group's partials in item order."""
    inp = synth.layer_inputs(203, 6, 1000 - 1000 % 8, 6208, 24, 48.0)
    a = run_layer(inp, fwd_only=True)
    for _ in range(3):
        b = run_layer(inp, fwd_only=True)
        for k in ("Y", "U"):
            assert torch.equal(a[k], b[k]), k


def test_adapter_b_zero(orc):
    # LoRA init of the lesson (B = 0): Y is the base product, dA is exactly zero
    inp = synth.layer_inputs(203, 64, 256, 512, 8, 16.0)
    inp.B[:] = 0
    out = run_layer(inp)
    assert torch.count_nonzero(out["dA"]).item() == 0
    check_full(orc, inp, out)


def test_all_zero_weight(orc):
    # W^ = 0: Y is the adapter term alone; the adapter has O(|Y|) weight here
    inp = synth.layer_inputs(204, 48, 128, 256, 8, 16.0, b_std=1.0)
    inp.W[:] = 0
    out = run_layer(inp)
    assert np.all(out["qw"].codes.cpu().numpy() == 0x77)
    check_full(orc, inp, out)


def test_adapter_term_dominant(orc):
    # B ~ N(0, 1): the LoRA term is of the order of |Y|, not hidden by the tolerance
    inp = synth.layer_inputs(205, 128, 256, 512, 16, 32.0, b_std=1.0)
    check_full(orc, inp, run_layer(inp))


def test_llama8b_attn(orc):
    c = synth.LLAMA8B_ATTN
    inp = synth.layer_inputs(c["id"], c["M"], c["N"], c["K"], c["r"], c["alpha"])
    out = run_layer(inp)
    rows = np.random.default_rng(0).choice(c["M"], 64, replace=False)
    check_full(orc, inp, out, rows=np.sort(rows))


@pytest.mark.parametrize("mat", [0, 2])
def test_llama8b_mlp(orc, mat):
    c = synth.LLAMA8B_MLP
    name, N, K = c["mats"][mat]
    inp = synth.layer_inputs(c["id"], c["M"], N, K, c["r"], c["alpha"], outliers="uniform", sub=mat)
    out = run_layer(inp)
    rows = np.sort(np.random.default_rng(1).choice(c["M"], 32, replace=False))
    check_full(orc, inp, out, rows=rows, jsel=[0, 37, 63])


@pytest.mark.parametrize("mat", [0, 1])
@pytest.mark.parametrize("M", [1, 8, 32])
def test_llama70b_decode(orc, M, mat):
    c = synth.LLAMA70B_DECODE
    name, N, K = c["mats"][mat]
    inp = synth.layer_inputs(c["id"], M, N, K, c["r"], c["alpha"], w_std=c["w_std"], sub=mat, with_grad=False)
    out = run_layer(inp, fwd_only=True)
    rows = np.arange(M) if M <= 8 else np.array([0, 5, 17, 31])
    check_full(orc, inp, out, rows=rows)


def test_graph_capture_replays_the_stream_results():
    """fwd + bwd captured in a CUDA graph (the library's side-stream fork/join becomes graph edges)
    and replayed: bit for bit the results of stream launches, for the CTA-pair path with two token
    tiles per unit and for the GEMV path."""
    for (M, N, K, r) in [(600, 520, 640, 16), (4, 264, 4160, 8)]:
        inp = synth.layer_inputs(206 + M, M, N, K, r, 2.0 * r)
        qw = q.nf4_quantize(torch.from_numpy(inp.W).cuda())
        X, A, B, G = (dev_bf16(t) for t in (inp.X, inp.A, inp.B, inp.G))
        Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        U = torch.empty((M, r), dtype=torch.bfloat16, device="cuda")
        dX = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
        dA = torch.empty((r, K), dtype=torch.float32, device="cuda")
        dB = torch.empty((N, r), dtype=torch.float32, device="cuda")
        wf = torch.empty(q.fwd_workspace_bytes(M, N, K, r), dtype=torch.uint8, device="cuda")
        wb = torch.empty(q.bwd_workspace_bytes(M, N, K, r), dtype=torch.uint8, device="cuda")

        def step():
            q.qlora_linear_fwd(qw, X, A, B, 2.0 * r, Y=Y, U_save=U, workspace=wf)
            q.qlora_linear_bwd(qw, X, A, B, 2.0 * r, G, U, dX=dX, dA=dA, dB=dB, workspace=wb)

        step()
        torch.cuda.synchronize()
        ref = [t.clone() for t in (Y, U, dX, dA, dB)]
        for t in (Y, U, dX, dA, dB):
            t.zero_()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                step()
        torch.cuda.current_stream().wait_stream(s)
        graph.replay()
        torch.cuda.synchronize()
        q.check_device_error()
        for name, a, b in zip(("Y", "U", "dX", "dA", "dB"), (Y, U, dX, dA, dB), ref):
            assert torch.equal(a, b), (M, name)


def test_concurrent_host_threads_on_their_own_streams():
    """Two host threads run fwd + bwd of different layers on their own streams at once: the
    library's side streams are shared per device (their enqueue is serialised), and every result
    equals that of the same call made alone."""
    import threading
    shapes = [(600, 520, 640, 16), (300, 264, 384, 8)]
    layers = []
    for i, (M, N, K, r) in enumerate(shapes):
        inp = synth.layer_inputs(220 + i, M, N, K, r, 2.0 * r)
        qw = q.nf4_quantize(torch.from_numpy(inp.W).cuda())
        X, A, B, G = (dev_bf16(t) for t in (inp.X, inp.A, inp.B, inp.G))
        layers.append((qw, X, A, B, G, 2.0 * r))
    torch.cuda.synchronize()

    def run(layer):
        qw, X, A, B, G, alpha = layer
        Y, U = q.qlora_linear_fwd(qw, X, A, B, alpha)
        dX, dA, dB = q.qlora_linear_bwd(qw, X, A, B, alpha, G, U)
        return [t for t in (Y, U, dX, dA, dB)]

    ref = [run(layer) for layer in layers]
    torch.cuda.synchronize()
    out = [None, None]
    errors = []

    def worker(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(20):
                    res = run(layers[i])
                s.synchronize()
            out[i] = res
        except Exception as e:  # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    q.check_device_error()
    for i in range(2):
        for a, b in zip(out[i], ref[i]):
            assert torch.equal(a, b), i
