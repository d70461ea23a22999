"""Seeded synthetic inputs for the QLoRA NF4 linear layer.

This module holds no arithmetic of the method: it only draws random numbers.  It is the one
module that both the CUDA path (bench, GPU tests) and the CPU oracle's tests use, so that both
sides see the same bytes.

Distributions follow the workloads the layer is measured on (weights ~ N(0, sigma) like the
pages' ``randn * 0.02``; activations and upstream gradients ~ N(0, 1); LoRA A with variance
1/K, LoRA B with std 0.01 so that the adapter path is exercised).  Host-side draws use numpy's
PCG64 with a fixed seed per (workload, tensor); bf16 tensors are the round-to-nearest-even
bf16 of an fp32 draw and are returned as uint16 bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 0x51A00000

# stream ids, one per tensor kind
S_W, S_X, S_A, S_B, S_G, S_OUT_MASK, S_OUT_VAL, S_OUT_SIGN = range(8)


def rng(workload_id: int, stream: int, sub: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(SEED_BASE + workload_id * 0x1000 + sub * 0x10 + stream))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (done by torch's dtype cast)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def normal_f32(g: np.random.Generator, shape, std: float) -> np.ndarray:
    return (g.standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def weight(workload_id: int, rows: int, cols: int, std: float, outliers: str | None = None,
           sub: int = 0) -> np.ndarray:
    """fp32 [rows, cols] ~ N(0, std), optionally with 0.1% outlier entries.

    outliers: None, "uniform" (value +-U(0.2, 1.0), fair sign) or "t3" (std * Student-t(3)).
    """
    w = normal_f32(rng(workload_id, S_W, sub), (rows, cols), std)
    if outliers:
        gm = rng(workload_id, S_OUT_MASK, sub)
        mask = gm.random(size=(rows, cols), dtype=np.float32) < np.float32(0.001)
        cnt = int(mask.sum())
        gv = rng(workload_id, S_OUT_VAL, sub)
        if outliers == "uniform":
            mag = gv.uniform(0.2, 1.0, size=cnt).astype(np.float32)
            sign = np.where(rng(workload_id, S_OUT_SIGN, sub).random(size=cnt) < 0.5, -1.0, 1.0).astype(np.float32)
            w[mask] = mag * sign
        elif outliers == "t3":
            w[mask] = (np.float32(std) * gv.standard_t(3, size=cnt)).astype(np.float32)
        else:
            raise ValueError(outliers)
    return w


@dataclass
class LayerInputs:
    """One linear layer's synthetic inputs (host copies)."""
    W: np.ndarray            # fp32 [N, K]
    X: np.ndarray            # bf16 bits [M, K]
    A: np.ndarray            # bf16 bits [r, K]
    B: np.ndarray            # bf16 bits [N, r]
    G: np.ndarray            # bf16 bits [M, N]
    r: int
    alpha: float
    meta: dict = field(default_factory=dict)

    @property
    def shape(self):
        return self.X.shape[0], self.W.shape[0], self.W.shape[1]


def layer_inputs(workload_id: int, M: int, N: int, K: int, r: int, alpha: float, w_std: float = 0.02,
                 outliers: str | None = None, sub: int = 0, b_std: float = 0.01, x_std: float = 1.0,
                 with_grad: bool = True) -> LayerInputs:
    W = weight(workload_id, N, K, w_std, outliers, sub)
    X = to_bf16_bits(normal_f32(rng(workload_id, S_X, sub), (M, K), x_std))
    A = to_bf16_bits(normal_f32(rng(workload_id, S_A, sub), (r, K), 1.0 / np.sqrt(K)))
    B = to_bf16_bits(normal_f32(rng(workload_id, S_B, sub), (N, r), b_std))
    G = (to_bf16_bits(normal_f32(rng(workload_id, S_G, sub), (M, N), 1.0)) if with_grad
         else np.zeros((0, N), dtype=np.uint16))
    return LayerInputs(W, X, A, B, G, r, alpha, dict(workload=workload_id, sub=sub))


# ---------------------------------------------------------------------------------------
# The measured workloads, by name and size.
# ---------------------------------------------------------------------------------------
TINY = dict(name="tiny-256x512-m16-r8", id=0, M=16, N=256, K=512, r=8, alpha=16.0)
LLAMA8B_ATTN = dict(name="llama3-8b-attn-proj-4096x4096-m4096-r16", id=1, M=4096, N=4096, K=4096, r=16, alpha=32.0)
LLAMA8B_MLP = dict(name="llama3-8b-mlp-4096<->14336-m8192-r64", id=2, M=8192, r=64, alpha=128.0,
                   mats=[("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336)])
LLAMA70B_DECODE = dict(name="llama70b-mlp-decode-8192<->28672-m{1,8,32}-r16", id=3, Ms=[1, 8, 32], r=16, alpha=32.0,
                       w_std=0.015, mats=[("up", 28672, 8192), ("down", 8192, 28672)])
LLAMA70B_SWEEP = dict(name="llama70b-80-layer-quantize-dequantize-sweep", id=4, layers=80, w_std=0.02,
                      mats=[("q", 8192, 8192), ("k", 1024, 8192), ("v", 1024, 8192), ("o", 8192, 8192),
                            ("gate", 28672, 8192), ("up", 28672, 8192), ("down", 8192, 28672)])
# Every adapter of Llama-3-8B with rank 16 on all seven linear layers of its 32 blocks (A [r, K]
# and B [N, r] per matrix): the parameters one optimizer step updates.
LLAMA8B_ADAPTERS = dict(name="llama3-8b-all-linear-adapters-r16-adamw", id=5, layers=32, r=16,
                        mats=[("q", 4096, 4096), ("k", 1024, 4096), ("v", 1024, 4096), ("o", 4096, 4096),
                              ("gate", 14336, 4096), ("up", 14336, 4096), ("down", 4096, 14336)])


def adapter_param_count(c=LLAMA8B_ADAPTERS) -> int:
    return c["layers"] * sum(c["r"] * (N + K) for _, N, K in c["mats"])


def tiny_inputs() -> LayerInputs:
    c = TINY
    return layer_inputs(c["id"], c["M"], c["N"], c["K"], c["r"], c["alpha"])


def sweep_weight_gpu(layer: int, mat_index: int, rows: int, cols: int, device="cuda", std: float = 0.02):
    """fp32 [rows, cols] on the GPU for the 80-layer sweep: N(0, std) plus 0.1% entries
    replaced by std * Student-t(3) (t = Z / sqrt(chi2_3 / 3)); drawn with torch's device
    generator seeded per (layer, matrix) so that any layer can be regenerated on its own."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(SEED_BASE + LLAMA70B_SWEEP["id"] * 0x1000 + layer * 0x10 + mat_index)
    w = torch.randn((rows, cols), generator=gen, device=device, dtype=torch.float32).mul_(std)
    mask = torch.rand((rows, cols), generator=gen, device=device) < 0.001
    cnt = int(mask.sum().item())
    if cnt:
        z = torch.randn(cnt, generator=gen, device=device)
        chi = torch.randn((cnt, 3), generator=gen, device=device).pow_(2).sum(1)
        w[mask] = std * z / torch.sqrt(chi / 3.0)
    return w


def normal_weight_gpu(workload_id: int, mat_index: int, rows: int, cols: int, std: float, device="cuda",
                      outliers: bool = False):
    """fp32 [rows, cols] ~ N(0, std) on the GPU (torch's seeded device generator, one stream per
    (workload, matrix)); with `outliers`, 0.1% of the entries replaced by +-U(0.2, 1.0) with a
    random sign (the MLP workload's outlier recipe)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(SEED_BASE + workload_id * 0x1000 + 0x800 + mat_index)
    w = torch.randn((rows, cols), generator=gen, device=device, dtype=torch.float32).mul_(std)
    if outliers:
        mask = torch.rand((rows, cols), generator=gen, device=device) < 0.001
        mag = torch.rand((rows, cols), generator=gen, device=device).mul_(0.8).add_(0.2)
        sign = torch.where(torch.rand((rows, cols), generator=gen, device=device) < 0.5, -1.0, 1.0)
        w = torch.where(mask, mag * sign, w)
    return w


# ---------------------------------------------------------------------------------------
# Optimizer-step inputs (flat fp32 arrays of adapter weights, gradients and AdamW moments).
# ---------------------------------------------------------------------------------------
S_P, S_GRAD, S_M, S_V = 16, 17, 18, 19


@dataclass
class OptimInputs:
    p: np.ndarray   # fp32 [n] weights
    g: np.ndarray   # fp32 [n] gradients
    m: np.ndarray   # fp32 [n] first moments
    v: np.ndarray   # fp32 [n] second moments (>= 0)


def adamw_inputs(workload_id: int, n: int, sub: int = 0) -> OptimInputs:
    """Weights: the first half A-like U(-1/64, 1/64), the rest B-like N(0, 0.01).  Gradients:
    N(0, 1e-3) times a log-normal(0, 1) per-element scale (a heavy tail), 1% exact zeros.  First
    moments N(0, 1e-4); second moments the square of N(0, 1e-3), 1% exact zeros (entries not yet
    updated)."""
    h = n // 2
    gp = rng(workload_id, S_P, sub)
    p = np.concatenate([gp.uniform(-1 / 64, 1 / 64, h), gp.standard_normal(n - h) * 0.01]).astype(np.float32)
    gg = rng(workload_id, S_GRAD, sub)
    g = (gg.standard_normal(n) * 1e-3 * np.exp(gg.standard_normal(n))).astype(np.float32)
    g[gg.random(n) < 0.01] = 0.0
    m = (rng(workload_id, S_M, sub).standard_normal(n) * 1e-4).astype(np.float32)
    gv = rng(workload_id, S_V, sub)
    v = np.square(gv.standard_normal(n) * 1e-3).astype(np.float32)
    v[gv.random(n) < 0.01] = 0.0
    return OptimInputs(p, g, m, v)


def adamw_inputs_gpu(workload_id: int, n: int, device="cuda"):
    """The distributions of adamw_inputs, drawn on the GPU with torch's seeded device generator
    (for sizes where host generation would dominate): returns (p, g, m, v) fp32 CUDA tensors."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(SEED_BASE + workload_id * 0x1000 + S_P)
    h = n // 2
    p = torch.empty(n, device=device, dtype=torch.float32)
    p[:h].uniform_(-1 / 64, 1 / 64, generator=gen)
    p[h:].normal_(0.0, 0.01, generator=gen)
    g = torch.randn(n, generator=gen, device=device).mul_(1e-3).mul_(torch.randn(n, generator=gen, device=device).exp_())
    g[torch.rand(n, generator=gen, device=device) < 0.01] = 0.0
    m = torch.randn(n, generator=gen, device=device).mul_(1e-4)
    v = torch.randn(n, generator=gen, device=device).mul_(1e-3).square_()
    v[torch.rand(n, generator=gen, device=device) < 0.01] = 0.0
    return p, g, m, v
