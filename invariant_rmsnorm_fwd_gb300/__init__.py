"""Batch-invariant RMSNorm forward/backward for GB300 (sm_103a).

Thin Python binding over the C ABI in include/rmsnorm_bi.h: every function
here marshals arguments and calls the library; every step of the computation
runs in the library's CUDA kernels.  There is no CPU path: if the library is
missing and cannot be built, importing the binding's functions raises.

PyTorch supplies device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

from . import layout  # noqa: F401  (host layout mapper)

_lib = None

OK = 0
ERR_NAMES = {
    -1: "NULL", -2: "HIDDEN", -3: "ALIGN", -4: "STRIDE", -5: "LAYOUT", -6: "WORKSPACE",
    -7: "PLAN", -8: "ID", -9: "DUPLICATE", -10: "CAPACITY", -11: "CUDA", -12: "DEVICE", -13: "VALUE",
}
STATUS_DOUBLE, STATUS_MISSING, STATUS_HEADER, STATUS_PLAN, STATUS_TIMEOUT = 1, 2, 4, 8, 16
PLAN_ITEM_BYTES = 528


class RmsNormError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = _load().rmsnorm_strerror(code).decode() if _lib is not None else str(code)
        super().__init__(f"{where}: {ERR_NAMES.get(code, code)} ({msg})")


class _Layout(ctypes.Structure):
    _fields_ = [
        ("n_tokens", ctypes.c_int64),
        ("rows_per_token", ctypes.c_int32),
        ("reserved0", ctypes.c_int32),
        ("token_stride", ctypes.c_int64),
        ("tok_id", ctypes.c_void_p),
        ("n_logical_tokens", ctypes.c_int64),
        ("plan", ctypes.c_void_p),
        ("plan_items", ctypes.c_int64),
    ]


def library_path() -> str:
    from . import _build
    return _build.LIB


def _load():
    """Load the CUDA library, building it in-tree first if it is absent or stale."""
    global _lib
    if _lib is not None:
        return _lib
    from . import _build
    path = _build.build()
    lib = ctypes.CDLL(path)
    P, I64, I32, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    LP = ctypes.POINTER(_Layout)
    sig = {
        "rmsnorm_fwd": ([P, P, I64, F, LP, P, P, P], ctypes.c_int),
        "rmsnorm_bwd_dx": ([P, P, P, I64, F, LP, P, P, P], ctypes.c_int),
        "rmsnorm_bwd_dweight_contrib": ([P, P, I64, F, LP, P, P], ctypes.c_int),
        "rmsnorm_dweight_workspace_bytes": ([I64, I64], ctypes.c_size_t),
        "rmsnorm_dweight_begin": ([P, ctypes.c_size_t, I64, I64, P], ctypes.c_int),
        "dweight_finalize": ([P, I64, I64, P, P], ctypes.c_int),
        "dweight_finalize_range": ([P, I64, I64, I64, I64, P, P], ctypes.c_int),
        "dweight_finalize_scaled": ([P, I64, I64, F, P, P], ctypes.c_int),
        "dweight_combine": ([P, I64, I64, F, P, P], ctypes.c_int),
        "rmsnorm_add_fwd": ([P, P, P, I64, F, LP, P, P, P, P], ctypes.c_int),
        "rmsnorm_add_bwd": ([P, P, P, P, I64, F, F, LP, P, P, P], ctypes.c_int),
        "rmsnorm_dweight_status": ([P, P, ctypes.POINTER(I32)], ctypes.c_int),
        "rmsnorm_plan_bytes": ([I64, I32, ctypes.POINTER(ctypes.c_size_t)], ctypes.c_int),
        "rmsnorm_plan_build": ([P, I64, I32, I64, P, ctypes.c_size_t, ctypes.POINTER(I64),
                                ctypes.POINTER(I64), ctypes.POINTER(I64)], ctypes.c_int),
        "rmsnorm_bwd_noalloc": ([P, P, P, I64, F, LP, P, P, P, P], ctypes.c_int),
        "gemm_dw_workspace_bytes": ([I64, I64, I64], ctypes.c_size_t),
        "gemm_dw_begin": ([P, ctypes.c_size_t, I64, I64, I64, P], ctypes.c_int),
        "gemm_dw_contrib": ([P, I64, P, I64, I64, I64, LP, P, P], ctypes.c_int),
        "gemm_dw_finalize": ([P, I64, I64, I64, F, P, P], ctypes.c_int),
        "gemm_dw_status": ([P, P, ctypes.POINTER(I32)], ctypes.c_int),
        "rmsnorm_strerror": ([ctypes.c_int], ctypes.c_char_p),
        "rmsnorm_kernel_launches": ([], I64),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _check(rc: int, where: str):
    if rc != OK:
        raise RmsNormError(rc, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def kernel_launches() -> int:
    return int(_load().rmsnorm_kernel_launches())


# ------------------------------------------------------------------ planning

def plan_capacity(n_tokens: int, rows_per_token: int) -> int:
    """Bytes of a plan buffer that always suffices for a call of n_tokens token slots."""
    cap = ctypes.c_size_t(0)
    _check(_load().rmsnorm_plan_bytes(int(n_tokens), int(rows_per_token), ctypes.byref(cap)), "rmsnorm_plan_bytes")
    return max(int(cap.value), PLAN_ITEM_BYTES)


def plan_build(tok_id: np.ndarray, rows_per_token: int, n_logical_tokens: int, out: np.ndarray = None):
    """Host planner (C++ in the library).  Returns (plan bytes as np.uint8, items,
    whole blocks, spilled rows).  `out` (contiguous np.uint8, e.g. a view of pinned
    memory) receives the plan in place; the returned bytes are then a view of it."""
    lib = _load()
    tok_id = np.ascontiguousarray(tok_id, dtype=np.int32)
    cap = ctypes.c_size_t(0)
    _check(lib.rmsnorm_plan_bytes(tok_id.size, rows_per_token, ctypes.byref(cap)), "rmsnorm_plan_bytes")
    if out is None:
        buf = np.empty(max(int(cap.value), PLAN_ITEM_BYTES), dtype=np.uint8)
    else:
        if out.dtype != np.uint8 or out.ndim != 1 or not out.flags["C_CONTIGUOUS"]:
            raise ValueError("plan_build: out must be a contiguous 1-D np.uint8 array")
        buf = out
    items, whole, spill = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
    _check(lib.rmsnorm_plan_build(tok_id.ctypes.data_as(ctypes.c_void_p), tok_id.size, rows_per_token,
                                  n_logical_tokens, buf.ctypes.data_as(ctypes.c_void_p), buf.size,
                                  ctypes.byref(items), ctypes.byref(whole), ctypes.byref(spill)),
           "rmsnorm_plan_build")
    return buf[:items.value * PLAN_ITEM_BYTES], items.value, whole.value, spill.value


@dataclass
class CallLayout:
    """Device-side descriptor of one call: token ids and (optionally) its plan."""
    tok_id: object                      # torch int32 [n_tokens] on the device
    plan: object                        # torch uint8 on the device, or None
    plan_items: int
    n_tokens: int
    rows_per_token: int
    n_logical_tokens: int
    whole_blocks: int = 0
    spill_rows: int = 0

    def struct(self, token_stride: int) -> _Layout:
        torch = _torch()
        if self.n_tokens:
            _cuda_tensor(self.tok_id, "layout.tok_id", torch.int32)
            if self.tok_id.numel() != self.n_tokens or not self.tok_id.is_contiguous():
                raise ValueError(f"layout.tok_id: expected {self.n_tokens} contiguous ids")
        if self.plan is not None and self.plan_items:
            _cuda_tensor(self.plan, "layout.plan", torch.uint8, self.tok_id.device)
            if self.plan.numel() < self.plan_items * PLAN_ITEM_BYTES or not self.plan.is_contiguous():
                raise ValueError(f"layout.plan: {self.plan_items} items need {self.plan_items * PLAN_ITEM_BYTES} "
                                 f"contiguous bytes")
        return _Layout(self.n_tokens, self.rows_per_token, 0, token_stride,
                       self.tok_id.data_ptr() if self.n_tokens else None,
                       self.n_logical_tokens,
                       self.plan.data_ptr() if self.plan is not None else None,
                       self.plan_items)


def call_layout(tok_id: np.ndarray, rows_per_token: int, n_logical_tokens: int, device="cuda",
                with_plan: bool = True) -> CallLayout:
    import torch
    tok_id = np.ascontiguousarray(tok_id, dtype=np.int32)
    tdev = torch.from_numpy(tok_id).to(device)
    plan = None
    items = whole = spill = 0
    if with_plan:
        pbytes, items, whole, spill = plan_build(tok_id, rows_per_token, n_logical_tokens)
        plan = torch.from_numpy(pbytes.copy()).to(device) if items else torch.zeros(16, dtype=torch.uint8,
                                                                                      device=device)
    return CallLayout(tdev, plan, items, tok_id.size, rows_per_token, n_logical_tokens, whole, spill)


# ------------------------------------------------------------------ ops

def _torch():
    import torch
    return torch


def _cuda_tensor(t, name: str, dtype, device=None):
    """Raise unless t is a CUDA tensor of `dtype` (on `device` when given): the
    library takes raw device pointers and cannot tell a host buffer or another
    element type from the right one."""
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor (got {t.device})")
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, the call's layout is on {device}")


def _rows_view(t, name: str, lay: "CallLayout", hidden: int) -> int:
    """Token stride (elements) of a bf16 [T, rows_per_token, hidden] or
    [T, rows_per_token * hidden] tensor whose first n_tokens token slots are the
    call's (T >= n_tokens; the library touches no slot past n_tokens)."""
    torch = _torch()
    _cuda_tensor(t, name, torch.bfloat16, lay.tok_id.device if lay.n_tokens else None)
    rpt = lay.rows_per_token
    if t.dim() == 3:
        ok = t.shape[1] == rpt and t.shape[2] == hidden and t.stride(2) == 1 and t.stride(1) == hidden
    elif t.dim() == 2:
        ok = t.shape[1] == rpt * hidden and t.stride(1) == 1
    else:
        ok = False
    if not ok:
        raise ValueError(f"{name}: expected [n_tokens, {rpt}, {hidden}] or [n_tokens, {rpt * hidden}] with "
                         f"unit column stride, got shape {tuple(t.shape)} strides {t.stride()}")
    if t.shape[0] < lay.n_tokens:
        raise ValueError(f"{name}: {t.shape[0]} token slots, the call's layout has {lay.n_tokens}")
    return t.stride(0)


def _same_stride(stride: int, *named):
    for name, t in named:
        if t is not None and t.stride(0) != stride:
            raise ValueError(f"{name}: token stride {t.stride(0)} differs from x's {stride} (one stride per call)")


def _weight(weight, lay: "CallLayout") -> int:
    torch = _torch()
    _cuda_tensor(weight, "weight", torch.bfloat16, lay.tok_id.device if lay.n_tokens else None)
    if weight.dim() != 1 or not weight.is_contiguous():
        raise ValueError(f"weight: expected a contiguous [hidden] tensor, got shape {tuple(weight.shape)}")
    return int(weight.shape[0])


def _f32_out(t, name: str, numel: int, device):
    torch = _torch()
    _cuda_tensor(t, name, torch.float32, device)
    if not t.is_contiguous() or t.numel() < numel:
        raise ValueError(f"{name}: expected a contiguous float32 tensor of at least {numel} elements")


def _workspace(ws, cls, device):
    if ws is None:
        return None
    if not isinstance(ws, cls):
        raise TypeError(f"workspace: expected {cls.__name__}, got {type(ws).__name__}")
    if device is not None and ws.buf.device != device:
        raise ValueError(f"workspace: on {ws.buf.device}, the call's layout is on {device}")
    return _ptr(ws.buf)


def rmsnorm_fwd(x, weight, lay: CallLayout, eps: float, y=None, rstd=None, stream=None):
    import torch
    H = _weight(weight, lay)
    stride = _rows_view(x, "x", lay, H)
    if y is None:
        y = torch.empty_like(x)
    _rows_view(y, "y", lay, H)
    _same_stride(stride, ("y", y))
    if rstd is not None:
        _f32_out(rstd, "rstd", lay.n_tokens * lay.rows_per_token, x.device)
    L = lay.struct(stride)
    _check(_load().rmsnorm_fwd(_ptr(x), _ptr(weight), H, eps, ctypes.byref(L), _ptr(y), _ptr(rstd),
                               _stream(stream)), "rmsnorm_fwd")
    return y


def rmsnorm_bwd_dx(x, weight, dy, lay: CallLayout, eps: float, dx=None, workspace=None, stream=None,
                   write_dx: bool = True):
    import torch
    H = _weight(weight, lay)
    stride = _rows_view(x, "x", lay, H)
    _rows_view(dy, "dy", lay, H)
    if dx is None and write_dx:
        dx = torch.empty_like(dy)
    if dx is not None:
        _rows_view(dx, "dx", lay, H)
    _same_stride(stride, ("dy", dy), ("dx", dx))
    ws = _workspace(workspace, DweightWorkspace, x.device)
    L = lay.struct(stride)
    _check(_load().rmsnorm_bwd_dx(_ptr(x), _ptr(weight), _ptr(dy), H, eps, ctypes.byref(L), _ptr(dx),
                                  ws, _stream(stream)), "rmsnorm_bwd_dx")
    return dx


def rmsnorm_add_fwd(x, residual, weight, lay: CallLayout, eps: float, h=None, y=None, rstd=None, stream=None):
    """Residual add fused with the norm: h = bf16(x + residual), y = RMSNorm(h) * w."""
    import torch
    H = _weight(weight, lay)
    stride = _rows_view(x, "x", lay, H)
    if h is None:
        h = torch.empty_like(x)
    if y is None:
        y = torch.empty_like(x)
    for name, t in (("residual", residual), ("h", h), ("y", y)):
        _rows_view(t, name, lay, H)
    _same_stride(stride, ("residual", residual), ("h", h), ("y", y))
    if rstd is not None:
        _f32_out(rstd, "rstd", lay.n_tokens * lay.rows_per_token, x.device)
    L = lay.struct(stride)
    _check(_load().rmsnorm_add_fwd(_ptr(x), _ptr(residual), _ptr(weight), H, eps, ctypes.byref(L), _ptr(h),
                                   _ptr(y), _ptr(rstd), _stream(stream)), "rmsnorm_add_fwd")
    return h, y


def rmsnorm_add_bwd(x, weight, dy, lay: CallLayout, eps: float, dres=None, grad_scale: float = 1.0, dx=None,
                    workspace=None, stream=None):
    """dx = bf16(grad_scale * (norm backward) + dres); x is the saved h.  The
    dweight contribution to `workspace` stays unscaled (scale it at finalize)."""
    import torch
    H = _weight(weight, lay)
    stride = _rows_view(x, "x", lay, H)
    _rows_view(dy, "dy", lay, H)
    if dx is None:
        dx = torch.empty_like(dy)
    _rows_view(dx, "dx", lay, H)
    if dres is not None:
        _rows_view(dres, "dres", lay, H)
    _same_stride(stride, ("dy", dy), ("dx", dx), ("dres", dres))
    ws = _workspace(workspace, DweightWorkspace, x.device)
    L = lay.struct(stride)
    _check(_load().rmsnorm_add_bwd(_ptr(x), _ptr(weight), _ptr(dy), _ptr(dres), H, eps, float(grad_scale),
                                   ctypes.byref(L), _ptr(dx), ws, _stream(stream)), "rmsnorm_add_bwd")
    return dx


def rmsnorm_bwd_dweight_contrib(x, dy, hidden: int, lay: CallLayout, eps: float, workspace, stream=None):
    stride = _rows_view(x, "x", lay, hidden)
    _rows_view(dy, "dy", lay, hidden)
    _same_stride(stride, ("dy", dy))
    if workspace is None:
        raise ValueError("workspace: required")
    ws = _workspace(workspace, DweightWorkspace, x.device)
    L = lay.struct(stride)
    _check(_load().rmsnorm_bwd_dweight_contrib(_ptr(x), _ptr(dy), hidden, eps, ctypes.byref(L), ws,
                                               _stream(stream)), "rmsnorm_bwd_dweight_contrib")


class DweightWorkspace:
    """Device workspace of one dweight reduction (allocated by PyTorch)."""

    def __init__(self, n_logical_rows: int, hidden: int, device="cuda"):
        import torch
        self.n_rows = int(n_logical_rows)
        self.hidden = int(hidden)
        self.bytes = int(_load().rmsnorm_dweight_workspace_bytes(self.n_rows, self.hidden))
        if self.bytes == 0:
            raise RmsNormError(-5, "rmsnorm_dweight_workspace_bytes")
        self.buf = torch.empty(self.bytes, dtype=torch.uint8, device=device)
        if self.buf.data_ptr() % 256:
            raise RuntimeError("workspace allocation is not 256-byte aligned")

    def begin(self, stream=None):
        _check(_load().rmsnorm_dweight_begin(_ptr(self.buf), self.bytes, self.n_rows, self.hidden,
                                             _stream(stream)), "rmsnorm_dweight_begin")

    def finalize(self, dweight=None, stream=None, grad_scale=None):
        """dweight of the reduction; with grad_scale the root is multiplied by it once."""
        import torch
        if dweight is None:
            dweight = torch.empty(self.hidden, dtype=torch.float32, device=self.buf.device)
        _f32_out(dweight, "dweight", self.hidden, self.buf.device)
        if grad_scale is None:
            _check(_load().dweight_finalize(_ptr(self.buf), self.n_rows, self.hidden, _ptr(dweight),
                                            _stream(stream)), "dweight_finalize")
        else:
            _check(_load().dweight_finalize_scaled(_ptr(self.buf), self.n_rows, self.hidden, float(grad_scale),
                                                   _ptr(dweight), _stream(stream)), "dweight_finalize_scaled")
        return dweight

    def finalize_range(self, block_lo: int, block_count: int, root=None, stream=None):
        """Node of the dweight tree over blocks [block_lo, block_lo + block_count)
        of this workspace (block_count a power of two, block_lo a multiple of it)."""
        import torch
        if root is None:
            root = torch.empty(self.hidden, dtype=torch.float32, device=self.buf.device)
        _f32_out(root, "root", self.hidden, self.buf.device)
        _check(_load().dweight_finalize_range(_ptr(self.buf), self.n_rows, self.hidden, int(block_lo),
                                              int(block_count), _ptr(root), _stream(stream)),
               "dweight_finalize_range")
        return root

    def status(self, stream=None) -> int:
        out = ctypes.c_int32(0)
        _check(_load().rmsnorm_dweight_status(_ptr(self.buf), _stream(stream), ctypes.byref(out)),
               "rmsnorm_dweight_status")
        return int(out.value)


def dweight_finalize(workspace: DweightWorkspace, dweight=None, stream=None):
    return workspace.finalize(dweight, stream)


def dweight_combine(roots, dweight=None, stream=None, grad_scale: float = 1.0):
    """Carry tree over FP32 roots [n, H] (device), the top of the dweight tree,
    the result multiplied once by grad_scale."""
    import torch
    _cuda_tensor(roots, "roots", torch.float32)
    if roots.dim() != 2 or not roots.is_contiguous():
        raise ValueError(f"roots: expected a contiguous [n, hidden] tensor, got shape {tuple(roots.shape)}")
    n, H = roots.shape
    if dweight is None:
        dweight = torch.empty(H, dtype=torch.float32, device=roots.device)
    _f32_out(dweight, "dweight", H, roots.device)
    _check(_load().dweight_combine(_ptr(roots), n, H, float(grad_scale), _ptr(dweight), _stream(stream)),
           "dweight_combine")
    return dweight


class GemmDwWorkspace:
    """Workspace of one deterministic linear-layer weight gradient (det_gemm dW)
    over n_logical_tokens tokens: logical-order copies of x and dy and a flag
    per token (see gemm_dw_* in the C header)."""

    def __init__(self, n_logical_tokens: int, in_features: int, out_features: int, device="cuda"):
        import torch
        self.n, self.i, self.o = int(n_logical_tokens), int(in_features), int(out_features)
        self.bytes = int(_load().gemm_dw_workspace_bytes(self.n, self.i, self.o))
        if self.bytes == 0:
            raise RmsNormError(-2, "gemm_dw_workspace_bytes")
        self.buf = torch.empty(self.bytes, dtype=torch.uint8, device=device)
        if self.buf.data_ptr() % 256:
            raise RuntimeError("workspace allocation is not 256-byte aligned")

    def begin(self, stream=None):
        _check(_load().gemm_dw_begin(_ptr(self.buf), self.bytes, self.n, self.i, self.o, _stream(stream)),
               "gemm_dw_begin")

    def contrib(self, x, dy, lay: CallLayout, stream=None):
        """Places one call's tokens: x [T, I] and dy [T, O] (row strides taken from the tensors)."""
        torch = _torch()
        dev = self.buf.device
        _cuda_tensor(x, "x", torch.bfloat16, dev)
        _cuda_tensor(dy, "dy", torch.bfloat16, dev)
        if not (x.dim() == 2 and dy.dim() == 2 and x.shape[1] == self.i and dy.shape[1] == self.o
                and x.stride(1) == 1 and dy.stride(1) == 1):
            raise ValueError(f"x [T, {self.i}] and dy [T, {self.o}] with unit column stride expected, got "
                             f"{tuple(x.shape)} / {tuple(dy.shape)}")
        if min(x.shape[0], dy.shape[0]) < lay.n_tokens:
            raise ValueError(f"x and dy hold {x.shape[0]} / {dy.shape[0]} token slots, the layout {lay.n_tokens}")
        if lay.n_tokens and lay.tok_id.device != dev:
            raise ValueError(f"layout on {lay.tok_id.device}, workspace on {dev}")
        L = lay.struct(x.stride(0))
        _check(_load().gemm_dw_contrib(_ptr(x), x.stride(0), _ptr(dy), dy.stride(0), self.i, self.o,
                                       ctypes.byref(L), _ptr(self.buf), _stream(stream)), "gemm_dw_contrib")

    def finalize(self, dw=None, grad_scale: float = 1.0, stream=None):
        import torch
        if dw is None:
            dw = torch.empty(self.o, self.i, dtype=torch.float32, device=self.buf.device)
        _f32_out(dw, "dw", self.o * self.i, self.buf.device)
        _check(_load().gemm_dw_finalize(_ptr(self.buf), self.n, self.i, self.o, float(grad_scale), _ptr(dw),
                                        _stream(stream)), "gemm_dw_finalize")
        return dw

    def status(self, stream=None) -> int:
        out = ctypes.c_int32(0)
        _check(_load().gemm_dw_status(_ptr(self.buf), _stream(stream), ctypes.byref(out)), "gemm_dw_status")
        return int(out.value)


NOALLOC_SCRATCH_BYTES = 16 << 20


def rmsnorm_bwd_noalloc(x, weight, dy, lay: CallLayout, eps: float, dx=None, dweight=None, status=None,
                        stream=None):
    """Backward with dweight for one call, using the library's built-in scratch
    instead of a workspace (see rmsnorm_bwd_noalloc in the C header)."""
    import torch
    H = _weight(weight, lay)
    stride = _rows_view(x, "x", lay, H)
    _rows_view(dy, "dy", lay, H)
    if dx is not None:
        _rows_view(dx, "dx", lay, H)
    _same_stride(stride, ("dy", dy), ("dx", dx))
    if dweight is None:
        dweight = torch.empty(H, dtype=torch.float32, device=x.device)
    _f32_out(dweight, "dweight", H, x.device)
    if status is not None:
        _cuda_tensor(status, "status", torch.int32, x.device)
    L = lay.struct(stride)
    _check(_load().rmsnorm_bwd_noalloc(_ptr(x), _ptr(weight), _ptr(dy), H, eps, ctypes.byref(L), _ptr(dx),
                                       _ptr(dweight), _ptr(status), _stream(stream)), "rmsnorm_bwd_noalloc")
    return dx, dweight
