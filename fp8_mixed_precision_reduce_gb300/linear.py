"""FP8Linear: a drop-in for torch.nn.Linear on the library's FP8 path.

The layer the pages build with te.Linear inside fp8_autocast ("Transformer
Engine으로 FP8 사용하기", the te.Linear(768, 768, bias=True) example under
"FP8 사용방안(recipe)", and its backward under "Backward Pass 처리"), under the
DelayedScaling recipe with the HYBRID format: E4M3 for the input and the
weight in the forward GEMM, E5M2 for the output gradient in dgrad and wgrad.

Every step of the layer is a call into libfp8mp (casts to row-major FP8
copies with their amaxes, the forward GEMM, the fused dgrad + wgrad launch
that reads those copies as they are, the fused bias gradient); this file only
allocates the outputs through torch and passes pointers. Like
sync_float8_amax_and_scale_history after backward in the pages' training
loop, ``update_scales()`` runs the delayed-scaling update of the layer's
four tensors (input, weight, output, output gradient) once per step.
"""

from __future__ import annotations

import torch

from . import (AMAX_MAX, E4M3, E5M2, Meta, delayed_scaling_update, fp8_linear_bwd_rowmajor, fp8_linear_fwd,
               fp8_quantize, fp8_quantize_dbias, fp8_quantize_dbias_workspace_bytes)

__all__ = ["FP8Linear"]


class _FP8LinearFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, weight, bias, layer):
        K = x.shape[-1]
        N = weight.shape[0]
        x2 = x.reshape(-1, K)
        if not x2.is_contiguous():
            x2 = x2.contiguous()
        M = x2.shape[0]
        dev = x.device
        u8 = torch.uint8
        X8 = torch.empty((M, K), dtype=u8, device=dev)
        W8 = torch.empty((N, K), dtype=u8, device=dev)
        # row-major copies only: the backward GEMMs read them along their rows
        fp8_quantize(x2, E4M3, layer.meta_x.scale, X8, None, layer.meta_x.cur_amax)
        fp8_quantize(weight.detach(), E4M3, layer.meta_w.scale, W8, None, layer.meta_w.cur_amax)
        y = torch.empty((M, N), dtype=x.dtype, device=dev)
        fp8_linear_fwd(X8, W8, layer.meta_x.scale_inv, layer.meta_w.scale_inv, y,
                       bias=bias.detach() if bias is not None else None, y_amax=layer.meta_y.cur_amax)
        # the codes were made with this step's scales: keep those for backward
        ctx.save_for_backward(X8, W8, layer.meta_x.scale_inv.clone(), layer.meta_w.scale_inv.clone())
        ctx.layer = layer
        ctx.shapes = (x.shape, x.dtype, weight.dtype, None if bias is None else bias.dtype)
        return y.reshape(*x.shape[:-1], N)

    @staticmethod
    def backward(ctx, dy):
        X8, W8, sinv_x, sinv_w = ctx.saved_tensors
        layer = ctx.layer
        x_shape, x_dtype, w_dtype, b_dtype = ctx.shapes
        M, K = X8.shape
        N = W8.shape[0]
        dy2 = dy.reshape(-1, N)
        if dy2.dtype != x_dtype:
            dy2 = dy2.to(x_dtype)
        if not dy2.is_contiguous():
            dy2 = dy2.contiguous()
        dev = dy.device
        D8 = torch.empty((M, N), dtype=torch.uint8, device=dev)
        md = layer.meta_dy
        db = None
        if b_dtype is not None and ctx.needs_input_grad[2]:
            db = torch.empty(N, dtype=b_dtype, device=dev)
            fp8_quantize_dbias(dy2, E5M2, md.scale, D8, None, db, layer.dbias_workspace(M, N), amax=md.cur_amax)
        else:
            fp8_quantize(dy2, E5M2, md.scale, D8, None, md.cur_amax)
        sinv_dy = md.scale_inv.clone()
        dx = torch.empty((M, K), dtype=x_dtype, device=dev) if ctx.needs_input_grad[0] else None
        dw = torch.empty((N, K), dtype=w_dtype, device=dev) if ctx.needs_input_grad[1] else None
        # dgrad and wgrad in one launch, from the row-major copies
        fp8_linear_bwd_rowmajor(D8, W8, X8, sinv_dy, sinv_w, sinv_x, dx, dw, dy_fmt=E5M2,
                                dw_nonfinite=layer.dw_nonfinite if dw is not None else None)
        return (dx.reshape(x_shape) if dx is not None else None), dw, db, None


class FP8Linear(torch.nn.Module):
    """y = x W^T + b with FP8 GEMMs under delayed scaling (HYBRID).

    in_features, out_features and the token count must be multiples of 16.
    The weight is kept in high precision (fp32 master or bf16) and cast to
    E4M3 every forward with the delayed scale; call update_scales() once per
    training step, after backward.
    """

    def __init__(self, in_features: int, out_features: int, bias: bool = True, history_len: int = 16,
                 amax_compute_algo: int = AMAX_MAX, margin: int = 0, device="cuda",
                 dtype: torch.dtype = torch.float32):
        super().__init__()
        if in_features % 16 or out_features % 16:
            raise ValueError("FP8 linears need in_features and out_features divisible by 16")
        self.in_features, self.out_features = in_features, out_features
        self.algo, self.margin = amax_compute_algo, margin
        bound = 1.0 / in_features ** 0.5
        self.weight = torch.nn.Parameter(
            torch.empty((out_features, in_features), device=device, dtype=dtype).uniform_(-bound, bound))
        self.bias = (torch.nn.Parameter(torch.empty(out_features, device=device, dtype=dtype).uniform_(-bound, bound))
                     if bias else None)
        self.meta_x = Meta(history_len, E4M3, device)
        self.meta_w = Meta(history_len, E4M3, device)
        self.meta_y = Meta(history_len, E4M3, device)
        self.meta_dy = Meta(history_len, E5M2, device)
        # 1 once a weight gradient of this layer held an Inf or NaN (ORed by
        # every backward); a master step given it as grad_nonfinite reads and
        # clears it instead of scanning the gradient again
        self.dw_nonfinite = torch.zeros(1, dtype=torch.int32, device=device)
        # the bias gradient's workspace: zero-filled once, and every call of
        # fp8_quantize_dbias leaves it zero, so it is reused without clearing
        self._dbias_ws = torch.zeros(0, dtype=torch.float32, device=device)

    def metas(self):
        return [self.meta_x, self.meta_w, self.meta_y, self.meta_dy]

    def dbias_workspace(self, rows: int, cols: int) -> torch.Tensor:
        """The zero-filled workspace of the bias-gradient cast, grown when a
        larger shape needs more."""
        need = (fp8_quantize_dbias_workspace_bytes(rows, cols) + 3) // 4
        if self._dbias_ws.numel() < need:
            self._dbias_ws = torch.zeros(need, dtype=torch.float32, device=self._dbias_ws.device)
        return self._dbias_ws

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return _FP8LinearFn.apply(x, self.weight, self.bias, self)

    def update_scales(self) -> None:
        """Roll the amax histories and refresh the scales for the next step."""
        delayed_scaling_update(self.metas(), self.algo, self.margin)
