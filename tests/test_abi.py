"""The C-ABI library loads and exports every entry point that the header
declares; host-side argument checks run without a GPU."""
import ctypes
import os
import re

import pytest

import invariant_rmsnorm_fwd_gb300 as rb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("rmsnorm_fwd", "rmsnorm_bwd_dx", "rmsnorm_bwd_dweight_contrib", "dweight_finalize",
              "rmsnorm_dweight_begin", "rmsnorm_dweight_workspace_bytes", "rmsnorm_plan_build"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(rb.library_path() if os.path.exists(rb.library_path()) else rb._load()._name)
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_no_atomic_accumulation_in_kernels():
    csrc = os.path.join(ROOT, "invariant_rmsnorm_fwd_gb300", "csrc")
    for f in os.listdir(csrc):
        assert "atomicAdd" not in open(os.path.join(csrc, f)).read(), f


def _layout(n_tokens=4, rpt=1, stride=8, tok=1):
    return rb._Layout(n_tokens, rpt, 0, stride, tok, 4, None, 0)


def test_host_side_errors_need_no_gpu():
    lib = rb._load()
    P = ctypes.c_void_p
    good = P(256)                                          # never dereferenced: checks fail first
    L = _layout()
    assert lib.rmsnorm_fwd(good, good, 12, 1e-6, ctypes.byref(L), good, None, None) == -2      # H % 8
    assert lib.rmsnorm_fwd(good, good, 24576, 1e-6, ctypes.byref(L), good, None, None) == -2   # too big
    assert lib.rmsnorm_fwd(good, good, 5128, 1e-6, ctypes.byref(_layout(stride=5128)), good, None, None) == -2
    assert lib.rmsnorm_fwd(good, good, 8200, 1e-6, ctypes.byref(_layout(stride=8200)), good, None, None) == -2
    assert lib.rmsnorm_fwd(good, good, 8, 1e-6, None, good, None, None) == -1
    assert lib.rmsnorm_fwd(None, good, 8, 1e-6, ctypes.byref(L), good, None, None) == -1
    assert lib.rmsnorm_fwd(P(258), good, 8, 1e-6, ctypes.byref(L), good, None, None) == -3
    assert lib.rmsnorm_fwd(good, good, 8, 1e-6, ctypes.byref(_layout(stride=12)), good, None, None) == -3
    assert lib.rmsnorm_fwd(good, good, 16, 1e-6, ctypes.byref(_layout(stride=8)), good, None, None) == -4
    assert lib.rmsnorm_fwd(good, good, 8, 1e-6, ctypes.byref(_layout(rpt=0)), good, None, None) == -5
    # dweight contribution without a plan
    assert lib.rmsnorm_bwd_dx(good, good, good, 8, 1e-6, ctypes.byref(L), good, good, None) == -7
    assert lib.rmsnorm_bwd_dweight_contrib(good, good, 8, 1e-6, ctypes.byref(L), None, None) == -1
    assert lib.rmsnorm_dweight_begin(good, 16, 64, 8, None) == -6
    assert lib.rmsnorm_dweight_begin(P(272), 1 << 20, 64, 8, None) == -3
    assert lib.dweight_finalize(good, 64, 8, None, None) == -1
    assert lib.rmsnorm_dweight_workspace_bytes(64, 12) == 0
    # an empty call is a no-op that needs no device
    assert lib.rmsnorm_fwd(good, good, 8, 1e-6, ctypes.byref(_layout(n_tokens=0, tok=None)), good, None, None) == 0
    # residual-add chain and loss-seed scale
    nan, inf = float("nan"), float("inf")
    assert lib.rmsnorm_add_fwd(good, None, good, 8, 1e-6, ctypes.byref(L), good, good, None, None) == -1
    assert lib.rmsnorm_add_fwd(good, good, good, 8, 1e-6, ctypes.byref(L), good, good, None, None) == -5   # h == y
    assert lib.rmsnorm_add_fwd(good, P(264), good, 8, 1e-6, ctypes.byref(L), good, P(512), None, None) == -3
    assert lib.rmsnorm_add_bwd(good, good, good, None, 8, 1e-6, nan, ctypes.byref(L), good, None, None) == -13
    assert lib.rmsnorm_add_bwd(good, good, good, None, 8, 1e-6, inf, ctypes.byref(L), good, None, None) == -13
    assert lib.rmsnorm_add_bwd(good, good, good, good, 8, 1e-6, 1.0, ctypes.byref(L), None, good, None) == -1
    assert lib.rmsnorm_add_bwd(good, good, good, None, 8, 1e-6, 1.0, ctypes.byref(L), good, good, None) == -7
    assert lib.dweight_finalize_scaled(good, 64, 8, nan, good, None) == -13
    assert lib.dweight_combine(good, 2, 8, inf, good, None) == -13
    assert lib.dweight_combine(good, 2048, 8, 1.0, good, None) == -5
    assert lib.dweight_finalize_range(good, 640, 8, 1, 2, good, None) == -5    # not aligned
    assert lib.dweight_finalize_range(good, 640, 8, 0, 3, good, None) == -5    # not a power of two
    # linear-layer weight gradient
    assert lib.gemm_dw_workspace_bytes(10, 12, 8) == 0                           # in_features % 8
    assert lib.gemm_dw_workspace_bytes(10, 16, 8) >= 256 + 10 * 4 + 10 * 16 * 2 + 10 * 8 * 2
    assert lib.gemm_dw_begin(good, 16, 10, 16, 8, None) == -6
    assert lib.gemm_dw_begin(P(272), 1 << 20, 10, 16, 8, None) == -3
    assert lib.gemm_dw_contrib(good, 16, good, 8, 16, 8, ctypes.byref(_layout(rpt=2)), good, None) == -5
    assert lib.gemm_dw_contrib(good, 8, good, 8, 16, 8, ctypes.byref(L), good, None) == -4    # x stride < I
    assert lib.gemm_dw_finalize(good, 10, 16, 8, nan, good, None) == -13
    assert lib.gemm_dw_finalize(None, 10, 16, 8, 1.0, good, None) == -1


def test_workspace_size_formula():
    lib = rb._load()
    n, h = 1000, 128
    b = lib.rmsnorm_dweight_workspace_bytes(n, h)
    nb = (n + 63) // 64
    assert b >= 256 + nb + n + nb * h * 4 + n * h * 4
    assert b % 256 == 0


def test_strerror_covers_codes():
    lib = rb._load()
    for c in range(0, -14, -1):
        assert lib.rmsnorm_strerror(c) not in (None, b"unknown error")
