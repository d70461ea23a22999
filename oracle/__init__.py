"""CPU oracle for the QLoRA NF4 frozen-base linear layer -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import this package.  The CUDA library never imports, links or calls it,
and this package shares no code, header or table with the CUDA library.

The arithmetic lives in ``nf4_oracle.c`` (plain C, fp32 where the pages' torch code is fp32,
fp64 for the layer products); this module only builds it with gcc and marshals numpy arrays
through ctypes.  Every function cites the page passage it restates in the C source.

Parity status: every function is pinned by ``tests/test_oracle_pins.py`` (worked examples,
closed forms, library special cases, brute force); nothing here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nf4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile nf4_oracle.c with gcc (-ffp-contract=off: no implicit fused multiply-add)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    """The compiled oracle; ORACLE_LIB names another build of nf4_oracle.c to load instead (the
    sanitizer test runs the pins against an AddressSanitizer / UBSan build that way)."""
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(os.environ.get("ORACLE_LIB") or build())
        _declare(_lib)
    return _lib


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_D = ctypes.c_double


def _declare(L):
    L.orc_norm_ppf.argtypes = [_D]
    L.orc_norm_ppf.restype = _D
    L.orc_nf4_levels.argtypes = [_P]
    L.orc_toy_levels.argtypes = [_D, _P]
    L.orc_int4_absmax.argtypes = [_P, _I64, _P, _P, _P]
    L.orc_blockwise_codes.argtypes = [_P, _I64, _I64, _P, ctypes.c_int, _P, _P]
    L.orc_blockwise_mse.argtypes = [_P, _I64, _I64, _P, ctypes.c_int]
    L.orc_blockwise_mse.restype = _D
    L.orc_pack_nibbles.argtypes = [_P, _I64, _P]
    L.orc_unpack_nibbles.argtypes = [_P, _I64, _P]
    L.orc_dq_mean.argtypes = [_P, _I64]
    L.orc_dq_mean.restype = ctypes.c_float
    L.orc_double_quant.argtypes = [_P, _I64, _P, _P, _P]
    L.orc_bf16_round.argtypes = [ctypes.c_float]
    L.orc_bf16_round.restype = ctypes.c_uint16
    L.orc_nf4_quantize.argtypes = [_P, _I64, _I64, _P, _P, _P, _P, _P]
    L.orc_dq_scale.argtypes = [ctypes.c_int8, ctypes.c_float, ctypes.c_float]
    L.orc_dq_scale.restype = ctypes.c_float
    L.orc_nf4_dequantize.argtypes = [_P, _P, _P, ctypes.c_float, _I64, _I64, _P]
    L.orc_layer_fwd_rows.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _D, _P, _I64, _P, _P]
    L.orc_layer_dx_rows.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _D, _P, _I64, _P]
    L.orc_layer_adapter_grads.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _D, _P, _P]
    L.orc_layer_adapter_grads_cols.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _D, _P, _I64, _P, _P]
    L.orc_nf4_storage_bytes.argtypes = [_I64, _I64]
    L.orc_nf4_storage_bytes.restype = _I64
    L.orc_bf16_round_d.argtypes = [_D]
    L.orc_bf16_round_d.restype = ctypes.c_uint16
    L.orc_merge.argtypes = [_P, _P, _P, _I64, _I64, _I64, _D, _P]
    L.orc_philox4x32_10.argtypes = [_P, _P, _P]
    L.orc_adamw_step.argtypes = [_P, _P, _P, _P, _I64, _D, _D, _D, _D, _D, _I64]
    L.orc_dropout_scale.argtypes = [ctypes.c_uint64, ctypes.c_uint64, _D, _I64, _P]
    L.orc_layer_fwd_rows_drop.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _D, _P, _P, _I64, _P, _P]
    L.orc_layer_dx_rows_drop.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _D, _P, _P, _I64, _P]
    L.orc_layer_adapter_grads_drop.argtypes = [_P, _P, _P, _P, _I64, _I64, _I64, _I64, _D, _P, _P, _P]


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


# ---------------------------------------------------------------------------------------
# Format constants and small building blocks
# ---------------------------------------------------------------------------------------

def norm_ppf(p: float) -> float:
    return lib().orc_norm_ppf(float(p))


def nf4_levels() -> np.ndarray:
    out = np.zeros(16, dtype=np.float32)
    lib().orc_nf4_levels(_ptr(out))
    return out


def toy_levels(d: float = 0.03) -> np.ndarray:
    out = np.zeros(16, dtype=np.float64)
    lib().orc_toy_levels(float(d), _ptr(out))
    return out


def int4_absmax(w: np.ndarray):
    w = _c(w, np.float32)
    codes = np.zeros(w.size, dtype=np.int32)
    w_hat = np.zeros(w.size, dtype=np.float32)
    am = ctypes.c_float(0.0)
    lib().orc_int4_absmax(_ptr(w), w.size, ctypes.byref(am), _ptr(codes), _ptr(w_hat))
    return float(am.value), codes, w_hat


def blockwise_codes(w: np.ndarray, bs: int, levels: np.ndarray):
    w = _c(w, np.float32).reshape(-1)
    levels = _c(levels, np.float32)
    codes = np.zeros(w.size, dtype=np.uint8)
    am = np.zeros(w.size // bs, dtype=np.float32)
    lib().orc_blockwise_codes(_ptr(w), w.size, bs, _ptr(levels), levels.size, _ptr(codes), _ptr(am))
    return codes, am


def blockwise_mse(w: np.ndarray, bs: int, levels: np.ndarray) -> float:
    w = _c(w, np.float32).reshape(-1)
    levels = _c(levels, np.float32)
    return lib().orc_blockwise_mse(_ptr(w), w.size, bs, _ptr(levels), levels.size)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    codes = _c(codes, np.uint8).reshape(-1)
    out = np.zeros(codes.size // 2, dtype=np.uint8)
    lib().orc_pack_nibbles(_ptr(codes), codes.size, _ptr(out))
    return out


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    packed = _c(packed, np.uint8).reshape(-1)
    out = np.zeros(packed.size * 2, dtype=np.uint8)
    lib().orc_unpack_nibbles(_ptr(packed), out.size, _ptr(out))
    return out


def dq_mean(s: np.ndarray) -> np.float32:
    s = _c(s, np.float32)
    return np.float32(lib().orc_dq_mean(_ptr(s), s.size))


def double_quant(s: np.ndarray):
    s = _c(s, np.float32)
    nb = s.size
    ng = (nb + 255) // 256
    q = np.zeros(nb, dtype=np.int8)
    c2 = np.zeros(ng, dtype=np.float32)
    mu = ctypes.c_float(0.0)
    lib().orc_double_quant(_ptr(s), nb, _ptr(q), _ptr(c2), ctypes.byref(mu))
    return q, c2, np.float32(mu.value)


def dq_scale(q: int, c2: float, mu: float) -> np.float32:
    return np.float32(lib().orc_dq_scale(int(q), float(c2), float(mu)))


def bf16_round(x: float) -> int:
    return int(lib().orc_bf16_round(float(np.float32(x))))


def bf16_round_array(x: np.ndarray) -> np.ndarray:
    f = lib().orc_bf16_round
    return np.array([f(float(v)) for v in _c(x, np.float32).reshape(-1)], dtype=np.uint16).reshape(np.shape(x))


def bf16_to_f64(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) to float64, exactly (a bf16 is the top half of an fp32)."""
    u = _c(h, np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------------------
# The quantized matrix and the layer
# ---------------------------------------------------------------------------------------

def nf4_quantize(W: np.ndarray):
    """Return dict(packed u8[n/2], qcode i8[nb], c2 f32[ng], mu f32, absmax f32[nb])."""
    W = _c(W, np.float32)
    rows, cols = W.shape
    n = rows * cols
    nb = n // 64
    ng = (nb + 255) // 256
    packed = np.zeros(n // 2, dtype=np.uint8)
    q = np.zeros(nb, dtype=np.int8)
    c2 = np.zeros(ng, dtype=np.float32)
    am = np.zeros(nb, dtype=np.float32)
    mu = ctypes.c_float(0.0)
    lib().orc_nf4_quantize(_ptr(W), rows, cols, _ptr(packed), _ptr(q), _ptr(c2), ctypes.byref(mu), _ptr(am))
    return dict(packed=packed, qcode=q, c2=c2, mu=np.float32(mu.value), absmax=am)


def nf4_dequantize(packed, qcode, c2, mu, rows: int, cols: int) -> np.ndarray:
    """bf16 bit patterns (uint16) of W^, shape [rows, cols]."""
    packed = _c(packed, np.uint8)
    qcode = _c(qcode, np.int8)
    c2 = _c(c2, np.float32)
    out = np.zeros(rows * cols, dtype=np.uint16)
    lib().orc_nf4_dequantize(_ptr(packed), _ptr(qcode), _ptr(c2), float(mu), rows, cols, _ptr(out))
    return out.reshape(rows, cols)


def layer_fwd_rows(What, X, A, B, alpha: float, rows=None):
    """fp64 Y[rows] and U[rows] from bf16 bit patterns What [N,K], X [M,K], A [r,K], B [N,r]."""
    What, X, A, B = (_c(t, np.uint16) for t in (What, X, A, B))
    N, K = What.shape
    M = X.shape[0]
    r = A.shape[0]
    sel = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    Y = np.zeros((sel.size, N), dtype=np.float64)
    U = np.zeros((sel.size, r), dtype=np.float64)
    lib().orc_layer_fwd_rows(_ptr(What), _ptr(X), _ptr(A), _ptr(B), M, N, K, r, float(alpha),
                             _ptr(sel), sel.size, _ptr(Y), _ptr(U))
    return Y, U


def layer_dx_rows(What, A, B, G, alpha: float, rows=None):
    """fp64 dX[rows] from bf16 bit patterns What [N,K], A [r,K], B [N,r], G [M,N]."""
    What, A, B, G = (_c(t, np.uint16) for t in (What, A, B, G))
    N, K = What.shape
    M = G.shape[0]
    r = A.shape[0]
    sel = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    dX = np.zeros((sel.size, K), dtype=np.float64)
    lib().orc_layer_dx_rows(_ptr(What), _ptr(A), _ptr(B), _ptr(G), M, N, K, r, float(alpha),
                            _ptr(sel), sel.size, _ptr(dX))
    return dX


def layer_adapter_grads(X, A, B, G, alpha: float):
    """fp64 dA [r,K] and dB [N,r] over all tokens."""
    X, A, B, G = (_c(t, np.uint16) for t in (X, A, B, G))
    M, K = X.shape
    N = G.shape[1]
    r = A.shape[0]
    dA = np.zeros((r, K), dtype=np.float64)
    dB = np.zeros((N, r), dtype=np.float64)
    lib().orc_layer_adapter_grads(_ptr(X), _ptr(A), _ptr(B), _ptr(G), M, N, K, r, float(alpha), _ptr(dA), _ptr(dB))
    return dA, dB


def layer_adapter_grads_cols(X, A, B, G, alpha: float, jsel):
    """fp64 dA[jsel, :] ([nj, K]) and dB[:, jsel]^T ([nj, N]) over all tokens."""
    X, A, B, G = (_c(t, np.uint16) for t in (X, A, B, G))
    M, K = X.shape
    N = G.shape[1]
    r = A.shape[0]
    js = _c(jsel, np.int64)
    dA = np.zeros((js.size, K), dtype=np.float64)
    dBt = np.zeros((js.size, N), dtype=np.float64)
    lib().orc_layer_adapter_grads_cols(_ptr(X), _ptr(A), _ptr(B), _ptr(G), M, N, K, r, float(alpha), _ptr(js), js.size,
                                       _ptr(dA), _ptr(dBt))
    return dA, dBt


def nf4_storage_bytes(rows: int, cols: int) -> int:
    return int(lib().orc_nf4_storage_bytes(rows, cols))


def bf16_round_d(x: float) -> int:
    """bf16 bit pattern of the fp64 value x, rounded once (nearest, ties to even)."""
    return int(lib().orc_bf16_round_d(float(x)))


def merge(What, A, B, alpha: float) -> np.ndarray:
    """bf16 bit patterns of W_m = bf16(W^ + (alpha/r) B A), shape [N, K], from bf16 bit patterns
    What [N, K], A [r, K], B [N, r]."""
    What, A, B = (_c(t, np.uint16) for t in (What, A, B))
    N, K = What.shape
    r = A.shape[0]
    out = np.zeros((N, K), dtype=np.uint16)
    lib().orc_merge(_ptr(What), _ptr(A), _ptr(B), N, K, r, float(alpha), _ptr(out))
    return out


def philox4x32_10(ctr, key) -> np.ndarray:
    """Philox4x32-10 block: four uint32 counter words and two uint32 key words -> four words."""
    c = _c(np.asarray(ctr, dtype=np.uint64).astype(np.uint32), np.uint32)
    k = _c(np.asarray(key, dtype=np.uint64).astype(np.uint32), np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def dropout_scale(seed: int, offset: int, p: float, M: int, K: int) -> np.ndarray:
    """fp64 [M, K]: 1 / (1 - p) where the element of the adapter input is kept, else 0."""
    D = np.zeros(M * K, dtype=np.float64)
    lib().orc_dropout_scale(ctypes.c_uint64(seed), ctypes.c_uint64(offset), float(p), M * K, _ptr(D))
    return D.reshape(M, K)


def layer_fwd_rows_drop(What, X, A, B, alpha: float, D, rows=None):
    What, X, A, B = (_c(t, np.uint16) for t in (What, X, A, B))
    D = _c(D, np.float64)
    N, K = What.shape
    M = X.shape[0]
    r = A.shape[0]
    sel = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    Y = np.zeros((sel.size, N), dtype=np.float64)
    U = np.zeros((sel.size, r), dtype=np.float64)
    lib().orc_layer_fwd_rows_drop(_ptr(What), _ptr(X), _ptr(A), _ptr(B), M, N, K, r, float(alpha), _ptr(D),
                                  _ptr(sel), sel.size, _ptr(Y), _ptr(U))
    return Y, U


def layer_dx_rows_drop(What, A, B, G, alpha: float, D, rows=None):
    What, A, B, G = (_c(t, np.uint16) for t in (What, A, B, G))
    D = _c(D, np.float64)
    N, K = What.shape
    M = G.shape[0]
    r = A.shape[0]
    sel = np.arange(M, dtype=np.int64) if rows is None else _c(rows, np.int64)
    dX = np.zeros((sel.size, K), dtype=np.float64)
    lib().orc_layer_dx_rows_drop(_ptr(What), _ptr(A), _ptr(B), _ptr(G), M, N, K, r, float(alpha), _ptr(D),
                                 _ptr(sel), sel.size, _ptr(dX))
    return dX


def layer_adapter_grads_drop(X, A, B, G, alpha: float, D):
    X, A, B, G = (_c(t, np.uint16) for t in (X, A, B, G))
    D = _c(D, np.float64)
    M, K = X.shape
    N = G.shape[1]
    r = A.shape[0]
    dA = np.zeros((r, K), dtype=np.float64)
    dB = np.zeros((N, r), dtype=np.float64)
    lib().orc_layer_adapter_grads_drop(_ptr(X), _ptr(A), _ptr(B), _ptr(G), M, N, K, r, float(alpha), _ptr(D),
                                       _ptr(dA), _ptr(dB))
    return dA, dB


def adamw_step(p, g, m, v, lr: float, b1: float, b2: float, eps: float, wd: float, t: int):
    """One AdamW step in fp64: returns new (p, m, v)."""
    p, g, m, v = (np.array(a, dtype=np.float64).ravel().copy() for a in (p, g, m, v))
    lib().orc_adamw_step(_ptr(p), _ptr(g), _ptr(m), _ptr(v), p.size, float(lr), float(b1), float(b2), float(eps),
                         float(wd), int(t))
    return p, m, v
