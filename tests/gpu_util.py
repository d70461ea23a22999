"""Helpers shared by the GPU parity tests: host<->device marshalling and the tolerance check."""
import numpy as np
import torch

import bit_nf4_quantized_36_b300 as q

# Acceptance for the fp32-accumulated layer outputs (relative Frobenius error and max-abs error
# relative to the largest reference magnitude), against the fp64 oracle.
REL_FRO = 5e-3
MAX_ABS_REL = 2e-2


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_close(name: str, got: np.ndarray, want: np.ndarray):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    den = np.linalg.norm(want)
    rel = np.linalg.norm(got - want) / den if den > 0 else np.linalg.norm(got)
    mx = np.abs(got - want).max() if got.size else 0.0
    ref_max = np.abs(want).max() if want.size else 0.0
    assert rel <= REL_FRO, f"{name}: relative Frobenius error {rel:.3e} > {REL_FRO}"
    assert mx <= MAX_ABS_REL * ref_max + 1e-30, f"{name}: max abs error {mx:.3e} > {MAX_ABS_REL} * {ref_max:.3e}"
    return rel, mx


def quantize_on_gpu(W: np.ndarray):
    qw = q.nf4_quantize(torch.from_numpy(np.ascontiguousarray(W, np.float32)).cuda())
    torch.cuda.synchronize()
    return qw


def nf4_to_host(qw):
    return dict(packed=qw.codes.cpu().numpy(), qcode=qw.scale_codes.cpu().numpy(), c2=qw.scale_scales.cpu().numpy(),
                mu=np.float32(qw.scale_offset.cpu().numpy()[0]))


def assert_nf4_equal(got: dict, want: dict):
    np.testing.assert_array_equal(got["packed"], want["packed"])
    np.testing.assert_array_equal(got["qcode"], want["qcode"])
    np.testing.assert_array_equal(got["c2"].view(np.uint32), want["c2"].view(np.uint32))
    assert np.float32(got["mu"]).view(np.uint32) == np.float32(want["mu"]).view(np.uint32)
