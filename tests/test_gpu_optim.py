"""GPU parity of the adapters' AdamW step over paged optimizer states (qlora_paged_* and
qlora_adamw_step) against the fp64 oracle ("QLoRA" glossary entry (ultralytics.com), "Como funciona
a QLoRA", paged-optimizers bullet; the update rule is AdamW, Loshchilov and Hutter).

Tolerance, from the kernel's fp32 arithmetic (u = 2^-24, every operation correctly rounded, the
coefficients rounded once from fp64):
  m' = fma(b1, m, (1-b1) g):            two roundings        -> |dm| <= 2u (b1|m| + (1-b1)|g|)
  v' = fma(b2, v, (1-b2) g g):          three roundings      -> |dv| <= 3u (b2 v + (1-b2) g^2)
  step = (lr/bc1) m' / (sqrt(v')/sqrt(bc2) + eps): the m' error divided by the denominator, plus
         about 8u relative from sqrt, the divisions, the product and the coefficients;
  p' = p (1 - lr wd) - step:            three more roundings of |p| and |step|.
Each bound is written below with a factor of 2 to 4 of margin.  The bf16 copy must equal the
round-to-nearest-even bf16 of the kernel's own fp32 result bit for bit."""
import ctypes

import numpy as np
import pytest
import torch

import bit_nf4_quantized_36_b300 as q
from bit_nf4_quantized_36_b300 import synth

pytestmark = pytest.mark.gpu

U = 2.0 ** -24
HP = dict(lr=2e-4, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01)


def _expect(orc, p, g, m, v, t, lr, betas, eps, weight_decay):
    """Oracle step in fp64 on the fp32 inputs, plus the per-element tolerances."""
    b1, b2 = (float(np.float32(b)) for b in betas)
    lr, eps, wd = float(np.float32(lr)), float(np.float32(eps)), float(np.float32(weight_decay))
    P, Mm, V = orc.adamw_step(p, g, m, v, lr, b1, b2, eps, wd, t)
    p64, g64, m64, v64 = (np.asarray(a, np.float64) for a in (p, g, m, v))
    bc1, bc2 = 1.0 - b1 ** t, 1.0 - b2 ** t
    denom = np.sqrt(V / bc2) + eps
    step = lr / bc1 * Mm / denom
    tol_m = 4 * U * (b1 * np.abs(m64) + (1 - b1) * np.abs(g64)) + 1e-45
    tol_v = 6 * U * (b2 * v64 + (1 - b2) * g64 * g64) + 1e-45
    tol_p = 16 * U * (np.abs(p64) + np.abs(step)) + lr / bc1 * tol_m / denom + 1e-45
    return P, Mm, V, tol_p, tol_m, tol_v


def _check(name, got, want, tol):
    err = np.abs(np.asarray(got, np.float64) - want)
    bad = np.flatnonzero(err > tol)
    assert bad.size == 0, (f"{name}: {bad.size} elements out of bound; first at {bad[0]}: got {got[bad[0]]!r}, "
                           f"want {want[bad[0]]!r}, tol {tol[bad[0]]:.3e}")


def _run(p, g, m, v, t, p_bf16=None, **hp):
    hp = {**HP, **hp}
    q.adamw_step(p, g, m, v, t, hp["lr"], hp["betas"], hp["eps"], hp["weight_decay"], p_bf16)
    torch.cuda.synchronize()


@pytest.mark.parametrize("n", [1, 3, 4, 7, 1024, 4 * 2048 * 148 + 5, 1 << 20])
def test_adamw_device_memory(orc, n):
    """Device arrays over several steps (each step checked from the kernel's own previous state);
    sizes cover the scalar tail only, one grid-stride pass and several."""
    inp = synth.adamw_inputs(70, n)
    p, g, m, v = (torch.from_numpy(a.copy()).cuda() for a in (inp.p, inp.g, inp.m, inp.v))
    pb = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    for t in (1, 2, 10):
        p0, m0, v0 = p.cpu().numpy(), m.cpu().numpy(), v.cpu().numpy()
        _run(p, g, m, v, t, pb)
        P, Mm, V, tp, tm, tv = _expect(orc, p0, inp.g, m0, v0, t, **HP)
        _check("m", m.cpu().numpy(), Mm, tm)
        _check("v", v.cpu().numpy(), V, tv)
        _check("p", p.cpu().numpy(), P, tp)
        pbits = pb.view(torch.int16).cpu().numpy().view(np.uint16)
        if n <= 65536:
            np.testing.assert_array_equal(pbits, orc.bf16_round_array(p.cpu().numpy()))
        else:
            assert torch.equal(pb, p.to(torch.bfloat16))


def test_adamw_special_cases(orc):
    """lr = 0 leaves p unchanged bit for bit; g = 0 with m = v = 0 leaves m, v at zero and only
    decays p; beta1 = beta2 = 0 makes the step lr g / (|g| + eps) whatever the old moments."""
    n = 4096
    inp = synth.adamw_inputs(71, n)
    p, g, m, v = (torch.from_numpy(a.copy()).cuda() for a in (inp.p, inp.g, inp.m, inp.v))
    _run(p, g, m, v, 3, lr=0.0)
    np.testing.assert_array_equal(p.cpu().numpy(), inp.p)
    z = torch.zeros(n, device="cuda")
    p = torch.from_numpy(inp.p.copy()).cuda()
    m, v = z.clone(), z.clone()
    _run(p, z, m, v, 1, weight_decay=0.0)
    np.testing.assert_array_equal(p.cpu().numpy(), inp.p)
    assert not m.any() and not v.any()
    p, m, v = (torch.from_numpy(a.copy()).cuda() for a in (inp.p, inp.m, inp.v))
    _run(p, torch.from_numpy(inp.g).cuda(), m, v, 5, betas=(0.0, 0.0), weight_decay=0.0, lr=1e-3)
    g64 = inp.g.astype(np.float64)
    want = inp.p - 1e-3 * g64 / (np.abs(g64) + 1e-8)
    np.testing.assert_allclose(p.cpu().numpy(), want, rtol=0, atol=1e-3 * 8 * U + 4 * U * np.abs(want).max())


def test_adamw_paged_states_wherever_the_pages_are(orc):
    """m and v in paged memory: a step with the pages on the host (migrated on demand), a step
    after paging them in, and a host read after paging them out give the device-memory result
    bit for bit; the results match the oracle."""
    n = (1 << 20) + 12
    inp = synth.adamw_inputs(72, n)
    ref_p, ref_m, ref_v = (torch.from_numpy(a.copy()).cuda() for a in (inp.p, inp.m, inp.v))
    g = torch.from_numpy(inp.g).cuda()
    opt = q.PagedAdamW(n, **HP)
    ctypes.memmove(opt.m.ptr, inp.m.ctypes.data, 4 * n)   # pages first touched on the host
    ctypes.memmove(opt.v.ptr, inp.v.ctypes.data, 4 * n)
    p = torch.from_numpy(inp.p.copy()).cuda()
    for t in (1, 2, 3):
        if t == 2:
            opt.page_in()
        if t == 3:
            opt.page_out()      # the step must fault the pages back in
        opt.step(p, g)
        _run(ref_p, g, ref_m, ref_v, t)
        np.testing.assert_array_equal(p.cpu().numpy(), ref_p.cpu().numpy())
    opt.page_out()
    torch.cuda.synchronize()
    hm = np.ctypeslib.as_array(opt.m.host_view(n)).copy()
    hv = np.ctypeslib.as_array(opt.v.host_view(n)).copy()
    np.testing.assert_array_equal(hm, ref_m.cpu().numpy())
    np.testing.assert_array_equal(hv, ref_v.cpu().numpy())
    # the zero-copy CUDA view sees the same bytes
    np.testing.assert_array_equal(opt.m.tensor(torch.float32, n).cpu().numpy(), hm)
    # one more step from the host-resident state, checked against the oracle
    p0 = p.cpu().numpy()
    opt.step(p, g)
    torch.cuda.synchronize()
    P, Mm, V, tp, tm, tv = _expect(orc, p0, inp.g, hm, hv, 4, **HP)
    _check("p", p.cpu().numpy(), P, tp)
    _check("m", np.ctypeslib.as_array(opt.m.host_view(n)), Mm, tm)
    _check("v", np.ctypeslib.as_array(opt.v.host_view(n)), V, tv)


def test_adamw_empty_and_buffer_errors():
    z = torch.zeros(0, device="cuda")
    q.adamw_step(z, z, z, z, 1, 1e-3)          # n = 0: no launch, no error
    small = q.PagedBuffer(64)
    with pytest.raises(ValueError):
        q.adamw_step(torch.zeros(32, device="cuda"), torch.zeros(32, device="cuda"), small, small, 1, 1e-3)
    with pytest.raises(q.QLoRAError):
        q._check(q._lib.load().qlora_paged_free(ctypes.c_void_p(torch.zeros(4, device="cuda").data_ptr())),
                 "free of device memory")
    small.free()


def test_adamw_llama8b_adapters_full_size(orc):
    """The whole adapter set of Llama-3-8B with rank 16 on every linear layer (41.9 M weights) in
    one launch, states paged and paged in, as the benchmark times it; 200,000 sampled elements
    against the oracle and the bf16 copy checked everywhere against the fp32 result."""
    n = synth.adapter_param_count()
    p, g, m0, v0 = synth.adamw_inputs_gpu(73, n)
    opt = q.PagedAdamW(n, **HP)
    opt.m.tensor(torch.float32, n).copy_(m0)
    opt.v.tensor(torch.float32, n).copy_(v0)
    opt.page_in()
    idx = np.sort(np.random.default_rng(5).choice(n, 200_000, replace=False))
    ti = torch.from_numpy(idx).cuda()
    p_s, g_s, m_s, v_s = (x[ti].cpu().numpy() for x in (p, g, m0, v0))
    del m0, v0
    pb = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    opt.step(p, g, pb)
    torch.cuda.synchronize()
    q.check_device_error()
    P, Mm, V, tp, tm, tv = _expect(orc, p_s, g_s, m_s, v_s, 1, **HP)
    _check("p", p[ti].cpu().numpy(), P, tp)
    _check("m", opt.m.tensor(torch.float32, n)[ti].cpu().numpy(), Mm, tm)
    _check("v", opt.v.tensor(torch.float32, n)[ti].cpu().numpy(), V, tv)
    assert torch.equal(pb, p.to(torch.bfloat16))
