"""Trainer-side asymmetric QAT (W4A16) of QUADS §3.2.

Eq. (12): the learner's forward multiplies bf16 activations by W-hat = QDQ_W(W), the weight
fake-quantized by the same quantizer the rollout uses (`weight_qdq`: its codes and scales are the
rollout's bit for bit, so Eq. (16)'s weight mismatch is exactly zero).  Eq. (13): the backward
pass treats the QDQ node as the identity for the weight (straight-through estimator) and
propagates the activation gradient through W-hat.  The optimizer keeps updating the bf16 master
weights.  The two GEMMs of a step are plain bf16 library GEMMs (cuBLAS through torch).
"""
from __future__ import annotations

import torch

from . import _lib as L
from .layers import Operand


def qdq_weight(w: torch.Tensor) -> torch.Tensor:
    """W-hat = DQ(Q(W)) in bf16 for W [N, K] or [G, N, K] (one tensor scale per [N, K] tensor);
    N % 128 == 0, K % 16 == 0."""
    w3 = w.detach().contiguous()
    if w3.dim() == 2:
        w3 = w3.unsqueeze(0)
    G, N, K = w3.shape
    op = Operand.empty(G * N, K, 0, G, device=w.device)
    w_hat = torch.empty(G, N, K, dtype=torch.bfloat16, device=w.device)
    L.weight_qdq(w3, G, N, K, op.codes, op.sf, op.sf_cols, op.tscale, w_hat=w_hat, w_hat_dtype=L.NVQ_BF16)
    return w_hat.view_as(w)


class QDQLinearFunction(torch.autograd.Function):
    """y = x W-hat^T with W-hat = QDQ_W(W) (Eq. (12)); dL/dW = dL/dW-hat (STE) and
    dL/dx = dL/dy W-hat (Eq. (13), row-major form)."""

    @staticmethod
    def forward(ctx, x: torch.Tensor, w: torch.Tensor):
        w_hat = qdq_weight(w)
        ctx.save_for_backward(x, w_hat)
        return x @ w_hat.t()

    @staticmethod
    def backward(ctx, gy: torch.Tensor):
        x, w_hat = ctx.saved_tensors
        gx = gy @ w_hat if ctx.needs_input_grad[0] else None
        gw = None
        if ctx.needs_input_grad[1]:
            gw = gy.reshape(-1, gy.shape[-1]).t() @ x.reshape(-1, x.shape[-1])
        return gx, gw


class QATLinear(torch.nn.Module):
    """Linear layer of the learner with W4A16 QAT: bf16 master weight [out, in], bf16
    activations, the forward sees the rollout's discretized weight values."""

    def __init__(self, in_features: int, out_features: int, device="cuda"):
        super().__init__()
        self.weight = torch.nn.Parameter(
            torch.empty(out_features, in_features, dtype=torch.bfloat16, device=device).normal_(0.0, 0.02))

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return QDQLinearFunction.apply(x, self.weight)
