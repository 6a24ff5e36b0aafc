"""HSTU LayerNorm-Multiply-SiLU-Dropout (LMSD): thin binding over the C ABI
of ``include/hstu_lmsd.h`` (argument marshalling only; every step runs in the
library's CUDA kernels).  Mirrors the page's ``hstu_lmsd_forward`` /
``hstu_lmsd_backward`` (page "HSTU LayerNorm-Multiply-SiLU-Dropout (LMSD)",
"Functions")."""
from __future__ import annotations

from ._lib import HstuError, library


def _stream(device):
    import torch
    return torch.cuda.current_stream(device).cuda_stream


def _rows(name, t, n, d):
    import torch
    if t.dtype != torch.bfloat16 or t.dim() != 2 or t.shape[0] != n or t.shape[1] != d:
        raise ValueError(f"{name}: expected bf16 ({n}, {d})")
    if t.stride(1) != 1:
        raise ValueError(f"{name}: the last dimension must be contiguous")


def hstu_lmsd_forward(x, u, weight, bias, eps: float = 1e-6, dropout_ratio: float = 0.0,
                      seed: int = 0, apply_u_silu: bool = True, concat_u: bool = True,
                      concat_x: bool = True):
    """Returns a dict: y_tensor (N, S*D) bf16, mean_tensor and rstd_tensor (N,)
    fp32, mask_tensor (N, D) int8 or None when dropout_ratio == 0."""
    import torch
    n, d = x.shape
    _rows("x", x, n, d)
    _rows("u", u, n, d)
    s = 1 + int(bool(concat_u)) + int(bool(concat_x))
    y = torch.empty(n, s * d, dtype=torch.bfloat16, device=x.device)
    mean = torch.empty(n, dtype=torch.float32, device=x.device)
    rstd = torch.empty(n, dtype=torch.float32, device=x.device)
    mask = torch.empty(n, d, dtype=torch.int8, device=x.device) if dropout_ratio > 0 else None
    st = library().hstu_lmsd_fwd(
        x.data_ptr(), x.stride(0), u.data_ptr(), u.stride(0), weight.data_ptr(), bias.data_ptr(),
        n, d, float(eps), float(dropout_ratio), int(bool(apply_u_silu)), int(bool(concat_u)),
        int(bool(concat_x)), int(seed), y.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
        mask.data_ptr() if mask is not None else None, _stream(x.device))
    if st != 0:
        raise HstuError(st)
    return {"y_tensor": y, "mean_tensor": mean, "rstd_tensor": rstd, "mask_tensor": mask}


def hstu_lmsd_backward(dy, x, u, weight, bias, mean, rstd, mask, dropout_ratio: float = 0.0,
                       apply_u_silu: bool = True, concat_u: bool = True, concat_x: bool = True,
                       compute_dweight: bool = True, dx=None, du=None, workspace=None):
    """Returns a dict: dx_tensor, du_tensor (N, D), dweight_tensor (D,) or None,
    dbias_tensor (D,), all bf16."""
    import torch
    n, d = x.shape
    lib = library()
    dx = torch.empty(n, d, dtype=torch.bfloat16, device=x.device) if dx is None else dx
    du = torch.empty(n, d, dtype=torch.bfloat16, device=x.device) if du is None else du
    dw = torch.empty(d, dtype=torch.bfloat16, device=x.device) if compute_dweight else None
    db = torch.empty(d, dtype=torch.bfloat16, device=x.device)
    need = lib.hstu_lmsd_bwd_workspace_size(n, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    st = lib.hstu_lmsd_bwd(
        dy.data_ptr(), dy.stride(0), x.data_ptr(), x.stride(0), u.data_ptr(), u.stride(0),
        weight.data_ptr(), bias.data_ptr(), mean.data_ptr(), rstd.data_ptr(),
        mask.data_ptr() if mask is not None else None, n, d, float(dropout_ratio),
        int(bool(apply_u_silu)), int(bool(concat_u)), int(bool(concat_x)),
        int(bool(compute_dweight)), dx.data_ptr(), dx.stride(0), du.data_ptr(), du.stride(0),
        dw.data_ptr() if dw is not None else None, db.data_ptr(), workspace.data_ptr(),
        workspace.numel(), _stream(x.device))
    if st != 0:
        raise HstuError(st)
    return {"dx_tensor": dx, "du_tensor": du, "dweight_tensor": dw, "dbias_tensor": db}
