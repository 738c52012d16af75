"""The binding refuses, before any library call, arguments that the C ABI
cannot check itself: host tensors, other element types, row counts
below the call's layout, mismatched token strides (CPU, no GPU needed)."""
import numpy as np
import pytest
import torch

import invariant_rmsnorm_fwd_gb300 as rb


def _layout(n=4, rpt=1, n_logical=4):
    tok = torch.arange(n, dtype=torch.int32)
    return rb.CallLayout(tok, None, 0, n, rpt, n_logical)


def test_host_tensors_and_wrong_types_are_refused():
    H = 16
    lay = _layout()
    x = torch.zeros(4, H, dtype=torch.bfloat16)
    w = torch.ones(H, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        rb.rmsnorm_fwd(x, w, lay, 1e-6)
    with pytest.raises(ValueError, match="CUDA tensor"):
        rb.rmsnorm_bwd_dx(x, w, x, lay, 1e-6)
    with pytest.raises(ValueError, match="CUDA tensor"):
        rb.rmsnorm_add_fwd(x, x, w, lay, 1e-6)
    with pytest.raises(ValueError, match="CUDA tensor"):
        rb.rmsnorm_add_bwd(x, w, x, lay, 1e-6)
    with pytest.raises(ValueError, match="CUDA tensor"):
        rb.rmsnorm_bwd_dweight_contrib(x, x, H, lay, 1e-6, workspace=None)
    with pytest.raises(ValueError, match="CUDA tensor"):
        rb.rmsnorm_bwd_noalloc(x, w, x, lay, 1e-6)
    with pytest.raises(ValueError, match="CUDA tensor"):
        rb.dweight_combine(torch.zeros(2, H))
    with pytest.raises(TypeError, match="torch.Tensor"):
        rb.dweight_combine(np.zeros((2, H), np.float32))
    with pytest.raises(TypeError, match="torch.Tensor"):
        rb.rmsnorm_fwd(x, np.ones(H, np.uint16), lay, 1e-6)


@pytest.fixture
def no_device_check(monkeypatch):
    """Let host tensors through the device check so that the shape checks behind
    it can be exercised on the CPU (every case below must still raise before the
    library is called)."""
    def check(t, name, dtype, device=None):
        if not isinstance(t, torch.Tensor):
            raise TypeError(name)
        if t.dtype != dtype:
            raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    monkeypatch.setattr(rb, "_cuda_tensor", check)


def test_shape_row_count_and_stride_checks(no_device_check):
    H = 16
    lay = _layout()
    w = torch.ones(H, dtype=torch.bfloat16)
    x = torch.zeros(4, H, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="token slots"):
        rb.rmsnorm_fwd(x[:3], w, lay, 1e-6)                       # fewer rows than the layout's slots
    with pytest.raises(ValueError, match="token slots"):
        rb.rmsnorm_bwd_dx(x, w, torch.zeros(3, H, dtype=torch.bfloat16), lay, 1e-6)
    with pytest.raises(ValueError, match="expected"):
        rb.rmsnorm_fwd(torch.zeros(4, H + 8, dtype=torch.bfloat16), w, lay, 1e-6)
    with pytest.raises(ValueError, match="expected"):
        rb.rmsnorm_fwd(torch.zeros(H, 4, dtype=torch.bfloat16).t(), w, lay, 1e-6)   # column stride 4
    with pytest.raises(TypeError, match="bfloat16"):
        rb.rmsnorm_fwd(x.float(), w, lay, 1e-6)
    with pytest.raises(ValueError, match="weight"):
        rb.rmsnorm_fwd(x, torch.ones(2, H // 2, dtype=torch.bfloat16), lay, 1e-6)
    wide = torch.zeros(4, 2 * H, dtype=torch.bfloat16)[:, :H]      # token stride 2H
    with pytest.raises(ValueError, match="token stride"):
        rb.rmsnorm_fwd(x, w, lay, 1e-6, y=wide)
    with pytest.raises(ValueError, match="rstd"):
        rb.rmsnorm_fwd(x, w, lay, 1e-6, y=x, rstd=torch.zeros(3))
    lay3 = _layout(rpt=2, n_logical=4)
    with pytest.raises(ValueError, match="expected"):
        rb.rmsnorm_fwd(torch.zeros(4, 3, H, dtype=torch.bfloat16), w, lay3, 1e-6)   # 3 heads, layout says 2
    with pytest.raises(TypeError, match="workspace"):
        rb.rmsnorm_bwd_dx(x, w, x, lay, 1e-6, workspace=object())
    with pytest.raises(ValueError, match="workspace"):
        rb.rmsnorm_bwd_dweight_contrib(x, x, H, lay, 1e-6, workspace=None)
    bad_ids = rb.CallLayout(torch.arange(4, dtype=torch.int64), None, 0, 4, 1, 4)
    with pytest.raises(TypeError, match="int32"):
        rb.rmsnorm_fwd(x, w, bad_ids, 1e-6)
