"""libqlora binding: the QLoRA NF4 frozen-base linear layer on B300.

Thin marshalling over the C ABI (include/qlora.h): torch is used for device memory and the
current CUDA stream only; every step of the layer runs in libqlora's CUDA kernels.  There is
no CPU or PyTorch fallback -- a missing library raises.

    q = nf4_quantize(W_fp32_cuda)                       # NF4 codes + double-quantized scales
    W_hat = nf4_dequantize(q)                           # bf16 [N, K]
    Y, U = qlora_linear_fwd(q, X, A, B, alpha)          # Y = X W^T + (alpha/r) X A^T B^T
    dX, dA, dB = qlora_linear_bwd(q, X, A, B, alpha, dY, U)
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib

__all__ = ["NF4Weight", "QLoRAError", "nf4_quantize", "nf4_quantize_noalloc", "nf4_dequantize", "qlora_linear_fwd", "qlora_linear_bwd",
           "qlora_merge", "qlora_linear_fwd_cat", "qlora_linear_bwd_cat", "qlora_linear_fwd_dropout",
           "qlora_linear_bwd_dropout", "nf4_storage_bytes", "quantize_workspace_bytes", "fwd_workspace_bytes", "bwd_workspace_bytes",
           "merge_workspace_bytes", "PagedBuffer", "PagedAdamW", "adamw_step",
           "check_device_error", "launch_count", "nf4_levels", "empty_nf4"]


class QLoRAError(RuntimeError):
    def __init__(self, status: int, what: str):
        name = _lib.QLORA_STATUS.get(status, str(status))
        super().__init__(f"{what}: {name} ({_lib.load().qlora_status_string(status).decode()})")
        self.status = status


def _check(status: int, what: str):
    if status != 0:
        raise QLoRAError(status, what)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _need(t: torch.Tensor, dtype, name: str, shape=None):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous CUDA tensor of dtype {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


@dataclass
class NF4Weight:
    """One NF4 matrix [rows, cols] with double-quantized block scales (device tensors)."""
    rows: int
    cols: int
    codes: torch.Tensor         # uint8 [rows*cols/2]
    scale_codes: torch.Tensor   # int8  [nb]
    scale_scales: torch.Tensor  # fp32  [ng]
    scale_offset: torch.Tensor  # fp32  [1]

    def struct(self) -> _lib.NF4TensorStruct:
        return _lib.NF4TensorStruct(self.rows, self.cols, self.codes.data_ptr(), self.scale_codes.data_ptr(),
                                    self.scale_scales.data_ptr(), self.scale_offset.data_ptr())

    @property
    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.codes, self.scale_codes, self.scale_scales,
                                                           self.scale_offset))


def nf4_storage_bytes(rows: int, cols: int) -> int:
    return int(_lib.load().qlora_nf4_storage_bytes(rows, cols))


def quantize_workspace_bytes(rows: int, cols: int) -> int:
    return int(_lib.load().qlora_quantize_workspace_bytes(rows, cols))


def fwd_workspace_bytes(M: int, N: int, K: int, r: int) -> int:
    return int(_lib.load().qlora_fwd_workspace_bytes(M, N, K, r))


def bwd_workspace_bytes(M: int, N: int, K: int, r: int) -> int:
    return int(_lib.load().qlora_bwd_workspace_bytes(M, N, K, r))


def merge_workspace_bytes(N: int, K: int, r: int) -> int:
    return int(_lib.load().qlora_merge_workspace_bytes(N, K, r))


def launch_count() -> int:
    return int(_lib.load().qlora_launch_count())


def nf4_levels() -> torch.Tensor:
    out = (ctypes.c_float * 16)()
    _lib.load().qlora_nf4_levels(ctypes.cast(out, ctypes.c_void_p))
    return torch.tensor(list(out), dtype=torch.float32)


def empty_nf4(rows: int, cols: int, device="cuda") -> NF4Weight:
    n = rows * cols
    nb = n // 64
    ng = (nb + 255) // 256
    return NF4Weight(rows, cols, torch.empty(n // 2, dtype=torch.uint8, device=device),
                     torch.empty(nb, dtype=torch.int8, device=device),
                     torch.empty(ng, dtype=torch.float32, device=device),
                     torch.empty(1, dtype=torch.float32, device=device))


def _workspace(nbytes: int, ws, device):
    if ws is not None:
        return ws
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


def nf4_quantize(W: torch.Tensor, out: NF4Weight | None = None, workspace: torch.Tensor | None = None,
                 stream=None) -> NF4Weight:
    """NF4-quantize fp32 W [N, K] (K % 64 == 0) with double-quantized scales."""
    _need(W, torch.float32, "W")
    rows, cols = W.shape
    if out is None:
        out = empty_nf4(rows, cols, W.device)
    L = _lib.load()
    need = int(L.qlora_quantize_workspace_bytes(rows, cols))
    if need == ctypes.c_size_t(-1).value:
        raise QLoRAError(2, "nf4_quantize")
    ws = _workspace(need, workspace, W.device)
    st = out.struct()
    _check(L.nf4_quantize(_ptr(W), ctypes.byref(st), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "nf4_quantize")
    return out


def nf4_quantize_noalloc(W: torch.Tensor, out: NF4Weight, stream=None) -> NF4Weight:
    """nf4_quantize with the library's fixed scratch area instead of a workspace (for callers that
    may not allocate device memory; rows * cols <= 2**28).  `out` must be preallocated."""
    _need(W, torch.float32, "W", (out.rows, out.cols))
    if out.codes.device != W.device:
        raise ValueError(f"nf4_quantize_noalloc: out is on {out.codes.device}, W on {W.device}")
    st = out.struct()
    # the library finds its scratch area on the current device: make that W's device
    with torch.cuda.device(W.device):
        _check(_lib.load().nf4_quantize_noalloc(_ptr(W), ctypes.byref(st), _stream(stream)), "nf4_quantize_noalloc")
    return out


def nf4_dequantize(q: NF4Weight, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """bf16 W^ [rows, cols] = bf16(NF4[c] * s'_b)."""
    if out is None:
        out = torch.empty((q.rows, q.cols), dtype=torch.bfloat16, device=q.codes.device)
    _need(out, torch.bfloat16, "out", (q.rows, q.cols))
    st = q.struct()
    _check(_lib.load().nf4_dequantize(ctypes.byref(st), _ptr(out), _stream(stream)), "nf4_dequantize")
    return out


def qlora_linear_fwd(q: NF4Weight, X: torch.Tensor, A: torch.Tensor, B: torch.Tensor, alpha: float,
                     Y: torch.Tensor | None = None, U_save: torch.Tensor | None = None, save_u: bool = True,
                     workspace: torch.Tensor | None = None, stream=None):
    """Y = X W^T + (alpha/r) (X A^T) B^T.  Returns (Y, U) with U = bf16((alpha/r) X A^T) or None."""
    M = X.shape[0]
    r = A.shape[0]
    _need(X, torch.bfloat16, "X", (M, q.cols))
    _need(A, torch.bfloat16, "A", (r, q.cols))
    _need(B, torch.bfloat16, "B", (q.rows, r))
    dev = X.device
    if Y is None:
        Y = torch.empty((M, q.rows), dtype=torch.bfloat16, device=dev)
    _need(Y, torch.bfloat16, "Y", (M, q.rows))
    if U_save is None and save_u:
        U_save = torch.empty((M, r), dtype=torch.bfloat16, device=dev)
    if U_save is not None:
        _need(U_save, torch.bfloat16, "U_save", (M, r))
    L = _lib.load()
    need = int(L.qlora_fwd_workspace_bytes(M, q.rows, q.cols, r))
    if need == ctypes.c_size_t(-1).value:
        raise QLoRAError(2, "qlora_linear_fwd")
    ws = _workspace(need, workspace, dev)
    st = q.struct()
    _check(L.qlora_linear_fwd(ctypes.byref(st), _ptr(X), M, _ptr(A), _ptr(B), r, float(alpha), _ptr(Y),
                              _ptr(U_save), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "qlora_linear_fwd")
    return Y, U_save


def qlora_linear_bwd(q: NF4Weight, X: torch.Tensor, A: torch.Tensor, B: torch.Tensor, alpha: float,
                     dY: torch.Tensor, U_saved: torch.Tensor | None = None, dX: torch.Tensor | None = None,
                     dA: torch.Tensor | None = None, dB: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None, stream=None):
    """Returns (dX bf16 [M, K], dA fp32 [r, K], dB fp32 [N, r])."""
    M = X.shape[0]
    r = A.shape[0]
    N, K = q.rows, q.cols
    _need(X, torch.bfloat16, "X", (M, K))
    _need(A, torch.bfloat16, "A", (r, K))
    _need(B, torch.bfloat16, "B", (N, r))
    _need(dY, torch.bfloat16, "dY", (M, N))
    if U_saved is not None:
        _need(U_saved, torch.bfloat16, "U_saved", (M, r))
    dev = X.device
    dX = torch.empty((M, K), dtype=torch.bfloat16, device=dev) if dX is None else dX
    dA = torch.empty((r, K), dtype=torch.float32, device=dev) if dA is None else dA
    dB = torch.empty((N, r), dtype=torch.float32, device=dev) if dB is None else dB
    _need(dX, torch.bfloat16, "dX", (M, K))
    _need(dA, torch.float32, "dA", (r, K))
    _need(dB, torch.float32, "dB", (N, r))
    L = _lib.load()
    need = int(L.qlora_bwd_workspace_bytes(M, N, K, r))
    if need == ctypes.c_size_t(-1).value:
        raise QLoRAError(2, "qlora_linear_bwd")
    ws = _workspace(need, workspace, dev)
    st = q.struct()
    _check(L.qlora_linear_bwd(ctypes.byref(st), _ptr(X), M, _ptr(A), _ptr(B), r, float(alpha), _ptr(dY),
                              _ptr(U_saved), _ptr(dX), _ptr(dA), _ptr(dB), _ptr(ws), ws.numel() * ws.element_size(),
                              _stream(stream)),
           "qlora_linear_bwd")
    return dX, dA, dB


def qlora_merge(q: NF4Weight, A: torch.Tensor, B: torch.Tensor, alpha: float, out: torch.Tensor | None = None,
                workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """bf16 W_m [rows, cols] = bf16(W^ + (alpha/r) B A): the adapters merged into the base weight."""
    r = A.shape[0]
    _need(A, torch.bfloat16, "A", (r, q.cols))
    _need(B, torch.bfloat16, "B", (q.rows, r))
    if out is None:
        out = torch.empty((q.rows, q.cols), dtype=torch.bfloat16, device=q.codes.device)
    _need(out, torch.bfloat16, "out", (q.rows, q.cols))
    L = _lib.load()
    need = int(L.qlora_merge_workspace_bytes(q.rows, q.cols, r))
    if need == ctypes.c_size_t(-1).value:
        raise QLoRAError(2, "qlora_merge")
    ws = _workspace(need, workspace, out.device)
    st = q.struct()
    _check(L.qlora_merge(ctypes.byref(st), _ptr(A), _ptr(B), r, float(alpha), _ptr(out), _ptr(ws),
                         ws.numel() * ws.element_size(), _stream(stream)), "qlora_merge")
    return out


def qlora_linear_fwd_dropout(q: NF4Weight, X: torch.Tensor, A: torch.Tensor, B: torch.Tensor, alpha: float, p: float,
                             seed: int, offset: int = 0, Y: torch.Tensor | None = None,
                             U_save: torch.Tensor | None = None, save_u: bool = True,
                             workspace: torch.Tensor | None = None, stream=None):
    """qlora_linear_fwd with LoRA dropout (probability p) on the adapter input; the mask is
    Philox4x32-10 of (seed, offset, element index).  Returns (Y, U)."""
    M = X.shape[0]
    r = A.shape[0]
    _need(X, torch.bfloat16, "X", (M, q.cols))
    _need(A, torch.bfloat16, "A", (r, q.cols))
    _need(B, torch.bfloat16, "B", (q.rows, r))
    dev = X.device
    if Y is None:
        Y = torch.empty((M, q.rows), dtype=torch.bfloat16, device=dev)
    _need(Y, torch.bfloat16, "Y", (M, q.rows))
    if U_save is None and save_u:
        U_save = torch.empty((M, r), dtype=torch.bfloat16, device=dev)
    L = _lib.load()
    need = int(L.qlora_fwd_dropout_workspace_bytes(M, q.rows, q.cols, r))
    if need == ctypes.c_size_t(-1).value:
        raise QLoRAError(2, "qlora_linear_fwd_dropout")
    ws = _workspace(need, workspace, dev)
    d = _lib.DropoutStruct(float(p), int(seed), int(offset))
    st = q.struct()
    _check(L.qlora_linear_fwd_dropout(ctypes.byref(st), _ptr(X), M, _ptr(A), _ptr(B), r, float(alpha), ctypes.byref(d),
                                      _ptr(Y), _ptr(U_save), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "qlora_linear_fwd_dropout")
    return Y, U_save


def qlora_linear_bwd_dropout(q: NF4Weight, X: torch.Tensor, A: torch.Tensor, B: torch.Tensor, alpha: float, p: float,
                             seed: int, dY: torch.Tensor, U_saved: torch.Tensor | None = None, offset: int = 0,
                             workspace: torch.Tensor | None = None, stream=None):
    """qlora_linear_bwd under the forward's dropout (same p, seed, offset).  Returns (dX, dA, dB)."""
    M = X.shape[0]
    r = A.shape[0]
    N, K = q.rows, q.cols
    _need(X, torch.bfloat16, "X", (M, K))
    _need(dY, torch.bfloat16, "dY", (M, N))
    if U_saved is not None:
        _need(U_saved, torch.bfloat16, "U_saved", (M, r))
    dev = X.device
    dX = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    dA = torch.empty((r, K), dtype=torch.float32, device=dev)
    dB = torch.empty((N, r), dtype=torch.float32, device=dev)
    L = _lib.load()
    need = int(L.qlora_bwd_dropout_workspace_bytes(M, N, K, r))
    if need == ctypes.c_size_t(-1).value:
        raise QLoRAError(2, "qlora_linear_bwd_dropout")
    ws = _workspace(need, workspace, dev)
    d = _lib.DropoutStruct(float(p), int(seed), int(offset))
    st = q.struct()
    _check(L.qlora_linear_bwd_dropout(ctypes.byref(st), _ptr(X), M, _ptr(A), _ptr(B), r, float(alpha), ctypes.byref(d),
                                      _ptr(dY), _ptr(U_saved), _ptr(dX), _ptr(dA), _ptr(dB), _ptr(ws),
                                      ws.numel() * ws.element_size(), _stream(stream)), "qlora_linear_bwd_dropout")
    return dX, dA, dB


class _CatModules:
    """ctypes view of a module list [(NF4Weight, A, B, alpha), ...] for the concatenated calls."""

    def __init__(self, modules):
        if not 1 <= len(modules) <= 4:
            raise ValueError("1 to 4 modules")
        self.structs = [m[0].struct() for m in modules]  # kept alive for the call
        arr = (_lib.CatModuleStruct * len(modules))()
        for i, (qw, A, B, alpha) in enumerate(modules):
            r = A.shape[0]
            _need(A, torch.bfloat16, f"A[{i}]", (r, qw.cols))
            _need(B, torch.bfloat16, f"B[{i}]", (qw.rows, r))
            arr[i].W = ctypes.pointer(self.structs[i])
            arr[i].A = A.data_ptr()
            arr[i].B = B.data_ptr()
            arr[i].r = r
            arr[i].alpha = float(alpha)
        self.arr = arr
        self.G = len(modules)
        self.N = (ctypes.c_int64 * self.G)(*[m[0].rows for m in modules])
        self.r = (ctypes.c_int32 * self.G)(*[m[1].shape[0] for m in modules])
        self.Ncat = sum(m[0].rows for m in modules)
        self.R8 = sum((m[1].shape[0] + 7) // 8 * 8 for m in modules)
        self.K = modules[0][0].cols


def qlora_linear_fwd_cat(modules, X: torch.Tensor, Y: torch.Tensor | None = None, U_save: torch.Tensor | None = None,
                         save_u: bool = True, workspace: torch.Tensor | None = None, stream=None):
    """Modules [(NF4Weight, A, B, alpha), ...] sharing X, as one N-concatenated layer.
    Returns (Y [M, sum N_i], U [M, R8] or None); Y[:, o_i:o_i + N_i] is module i's output."""
    cm = _CatModules(modules)
    M = X.shape[0]
    _need(X, torch.bfloat16, "X", (M, cm.K))
    dev = X.device
    if Y is None:
        Y = torch.empty((M, cm.Ncat), dtype=torch.bfloat16, device=dev)
    _need(Y, torch.bfloat16, "Y", (M, cm.Ncat))
    if U_save is None and save_u:
        U_save = torch.empty((M, cm.R8), dtype=torch.bfloat16, device=dev)
    if U_save is not None:
        _need(U_save, torch.bfloat16, "U_save", (M, cm.R8))
    L = _lib.load()
    need = int(L.qlora_cat_fwd_workspace_bytes(ctypes.cast(cm.N, ctypes.c_void_p), ctypes.cast(cm.r, ctypes.c_void_p),
                                               cm.G, M, cm.K))
    if need == ctypes.c_size_t(-1).value:
        raise QLoRAError(2, "qlora_linear_fwd_cat")
    ws = _workspace(need, workspace, dev)
    _check(L.qlora_linear_fwd_cat(ctypes.cast(cm.arr, ctypes.c_void_p), cm.G, _ptr(X), M, _ptr(Y), _ptr(U_save),
                                  _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "qlora_linear_fwd_cat")
    return Y, U_save


def qlora_linear_bwd_cat(modules, X: torch.Tensor, dY: torch.Tensor, U_saved: torch.Tensor | None = None,
                         dX: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None):
    """Returns (dX bf16 [M, K], [dA_i fp32 [r_i, K]], [dB_i fp32 [N_i, r_i]])."""
    cm = _CatModules(modules)
    M = X.shape[0]
    _need(X, torch.bfloat16, "X", (M, cm.K))
    _need(dY, torch.bfloat16, "dY", (M, cm.Ncat))
    if U_saved is not None:
        _need(U_saved, torch.bfloat16, "U_saved", (M, cm.R8))
    dev = X.device
    dX = torch.empty((M, cm.K), dtype=torch.bfloat16, device=dev) if dX is None else dX
    _need(dX, torch.bfloat16, "dX", (M, cm.K))
    dA = [torch.empty((m[1].shape[0], cm.K), dtype=torch.float32, device=dev) for m in modules]
    dB = [torch.empty((m[0].rows, m[1].shape[0]), dtype=torch.float32, device=dev) for m in modules]
    pa = (ctypes.c_void_p * cm.G)(*[t.data_ptr() for t in dA])
    pb = (ctypes.c_void_p * cm.G)(*[t.data_ptr() for t in dB])
    L = _lib.load()
    need = int(L.qlora_cat_bwd_workspace_bytes(ctypes.cast(cm.N, ctypes.c_void_p), ctypes.cast(cm.r, ctypes.c_void_p),
                                               cm.G, M, cm.K))
    if need == ctypes.c_size_t(-1).value:
        raise QLoRAError(2, "qlora_linear_bwd_cat")
    ws = _workspace(need, workspace, dev)
    _check(L.qlora_linear_bwd_cat(ctypes.cast(cm.arr, ctypes.c_void_p), cm.G, _ptr(X), M, _ptr(dY), _ptr(U_saved),
                                  _ptr(dX), ctypes.cast(pa, ctypes.c_void_p), ctypes.cast(pb, ctypes.c_void_p),
                                  _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "qlora_linear_bwd_cat")
    return dX, dA, dB


class PagedBuffer:
    """Unified (managed) memory from qlora_paged_alloc, for optimizer states that page to host RAM
    when GPU memory runs short.  Freed when the object and every tensor view of it are gone."""

    def __init__(self, nbytes: int):
        out = ctypes.c_void_p()
        _check(_lib.load().qlora_paged_alloc(int(nbytes), ctypes.byref(out)), "qlora_paged_alloc")
        self.ptr = int(out.value)
        self.nbytes = int(nbytes)

    def free(self) -> None:
        if self.ptr:
            _check(_lib.load().qlora_paged_free(ctypes.c_void_p(self.ptr)), "qlora_paged_free")
            self.ptr = 0

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass

    def prefetch(self, where="cuda", offset: int = 0, nbytes: int | None = None, stream=None) -> None:
        """Move the pages of [offset, offset + nbytes) to a device ("cuda", "cuda:i", an ordinal or a
        torch.device) or to host memory ("cpu"), asynchronously on `stream`."""
        nbytes = self.nbytes - offset if nbytes is None else nbytes
        if offset < 0 or nbytes < 0 or offset + nbytes > self.nbytes:
            raise ValueError("prefetch range outside the buffer")
        if where == "cpu":
            dev = _lib.QLORA_PAGE_HOST
        elif isinstance(where, int):
            dev = where
        else:
            d = torch.device(where)
            dev = d.index if d.index is not None else torch.cuda.current_device()
        _check(_lib.load().qlora_paged_prefetch(ctypes.c_void_p(self.ptr + offset), nbytes, dev, _stream(stream)),
               "qlora_paged_prefetch")

    def zero_(self) -> "PagedBuffer":
        """Zero-fill from the host (places untouched pages in host memory)."""
        ctypes.memset(self.ptr, 0, self.nbytes)
        return self

    def host_view(self, count: int | None = None, offset: int = 0, ctype=ctypes.c_float):
        """A host ctypes array over the buffer; valid to read only with no kernel in flight on it."""
        count = (self.nbytes - offset) // ctypes.sizeof(ctype) if count is None else count
        return (ctype * count).from_address(self.ptr + offset)

    def tensor(self, dtype=torch.float32, count: int | None = None, offset: int = 0) -> torch.Tensor:
        """A zero-copy 1-D CUDA tensor over the buffer (keeps the buffer alive)."""
        es = torch.empty((), dtype=dtype).element_size()
        count = (self.nbytes - offset) // es if count is None else count
        if offset < 0 or offset % es or offset + count * es > self.nbytes:
            raise ValueError("view outside the buffer")
        # bf16 has no array-interface type string: view 16-bit integers as bf16
        typestr = {torch.float32: "<f4", torch.bfloat16: "<i2", torch.int32: "<i4", torch.uint8: "|u1"}[dtype]
        buf = self

        class _View:
            __cuda_array_interface__ = {"shape": (count,), "typestr": typestr, "data": (self.ptr + offset, False),
                                        "version": 3, "strides": None}
            owner = buf

        t = torch.as_tensor(_View(), device=f"cuda:{torch.cuda.current_device()}")
        return t.view(torch.bfloat16) if dtype == torch.bfloat16 else t


def _f32_addr(x, n: int | None, name: str) -> tuple[int, int]:
    """(address, elements) of an fp32 array given as a CUDA tensor or a PagedBuffer."""
    if isinstance(x, PagedBuffer):
        cnt = x.nbytes // 4
        if n is not None and cnt < n:
            raise ValueError(f"{name}: paged buffer holds {cnt} fp32 elements, need {n}")
        return x.ptr, cnt if n is None else n
    _need(x, torch.float32, name)
    if n is not None and x.numel() != n:
        raise ValueError(f"{name} has {x.numel()} elements, expected {n}")
    return x.data_ptr(), x.numel()


def adamw_step(p, g, m, v, t: int, lr: float, betas=(0.9, 0.999), eps: float = 1e-8, weight_decay: float = 0.0,
               p_bf16: torch.Tensor | None = None, stream=None) -> None:
    """One AdamW step (qlora_adamw_step) on flat fp32 arrays: p, m, v updated in place, g read;
    p_bf16 (optional bf16 tensor) receives bf16(p).  Each array is a CUDA tensor or a PagedBuffer."""
    pa, n = _f32_addr(p, None, "p")
    ga, _ = _f32_addr(g, n, "g")
    ma, _ = _f32_addr(m, n, "m")
    va, _ = _f32_addr(v, n, "v")
    if p_bf16 is not None:
        _need(p_bf16, torch.bfloat16, "p_bf16")
        if p_bf16.numel() != n:
            raise ValueError(f"p_bf16 has {p_bf16.numel()} elements, expected {n}")
    hp = _lib.AdamWStruct(lr, betas[0], betas[1], eps, weight_decay)
    _check(_lib.load().qlora_adamw_step(ctypes.byref(hp), int(t), n, ctypes.c_void_p(pa), ctypes.c_void_p(ga),
                                        ctypes.c_void_p(ma), ctypes.c_void_p(va), _ptr(p_bf16), _stream(stream)),
           "qlora_adamw_step")


class PagedAdamW:
    """AdamW for the adapters with paged optimizer states: m and v (fp32, n each) live in unified
    memory.  page_out() moves them to host RAM before a memory spike, page_in() brings them back
    before the next step; step() is correct wherever the pages are."""

    def __init__(self, n: int, lr: float = 2e-4, betas=(0.9, 0.999), eps: float = 1e-8,
                 weight_decay: float = 0.0):
        self.n, self.lr, self.betas, self.eps, self.weight_decay = int(n), lr, betas, eps, weight_decay
        self.m = PagedBuffer(4 * self.n).zero_()
        self.v = PagedBuffer(4 * self.n).zero_()
        self.t = 0

    def page_out(self, stream=None) -> None:
        self.m.prefetch("cpu", stream=stream)
        self.v.prefetch("cpu", stream=stream)

    def page_in(self, device="cuda", stream=None) -> None:
        self.m.prefetch(device, stream=stream)
        self.v.prefetch(device, stream=stream)

    def step(self, p, g, p_bf16: torch.Tensor | None = None, stream=None) -> None:
        self.t += 1
        adamw_step(p, g, self.m, self.v, self.t, self.lr, self.betas, self.eps, self.weight_decay, p_bf16, stream)


def check_device_error(stream=None) -> None:
    _check(_lib.load().qlora_check_device_error(_stream(stream)), "device error word")


def test_inject(flags: int) -> None:
    """Failure-path test hook of the library (qlora_test_inject); 0 switches it off."""
    _check(_lib.load().qlora_test_inject(int(flags)), "test_inject")


test_inject.__test__ = False  # a library hook, not a pytest test
