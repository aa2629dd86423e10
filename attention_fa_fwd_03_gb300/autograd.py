"""Differentiable attention: a ``torch.autograd.Function`` over the C ABI.

Follows page "mlx-bun 0.0.4: package/src/model/flash-attention.ts", section
"Differentiable op: flash forward + manual backward via CustomVjp": the
forward returns O and keeps the per-row log-sum-exp L beside q, k, v and O;
the backward is the hand-written VJP (D-vector, dK/dV, dQ kernels), which
recomputes the probabilities from L instead of storing them. The cotangent of
L is discarded (L is marked non-differentiable here), as on that page.

Differences from the page: fp16 and bf16 both run natively (no cast to fp16
and back), and sliding windows run in the same kernels instead of falling
back to another attention op. Only argument marshalling happens here: output
and workspace tensors are allocated by PyTorch, every step of the computation
runs in the library's kernels, and there is no CPU path (a CPU tensor raises).

    from attention_fa_fwd_03_gb300.autograd import flash_attention
    o = flash_attention(q, k, v, causal=True)          # q [B,Hq,Tq,D], k/v [B,Hkv,Tkv,D]
    o.backward(do)                                      # fills q.grad, k.grad, v.grad
"""
from __future__ import annotations

import math

import torch

from . import fa_bwd, fa_bwd_workspace_size, fa_fwd

__all__ = ["FlashAttention", "flash_attention"]


class FlashAttention(torch.autograd.Function):
    """(q, k, v, scale, causal, window) -> (O, LSE); gradients for q, k, v only."""

    @staticmethod
    def forward(ctx, q, k, v, scale: float, causal: bool, window: int):
        with torch.cuda.device(q.device):
            o = torch.empty_like(q)
            lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
            fa_fwd(q, k, v, o, lse, scale, causal, window)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.attn = (scale, causal, window)
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, _dlse):
        q, k, v, o, lse = ctx.saved_tensors
        scale, causal, window = ctx.attn
        with torch.cuda.device(q.device):
            do = do.contiguous()
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
            ws = torch.empty(fa_bwd_workspace_size(*q.shape[:3]), dtype=torch.uint8,
                             device=q.device)
            fa_bwd(q, k, v, o, do, lse, dq, dk, dv, scale, causal, window, workspace=ws)
        return dq, dk, dv, None, None, None


def flash_attention(q, k, v, scale: float | None = None, causal: bool = False, window: int = 0,
                    return_lse: bool = False):
    """Exact attention O = softmax(s Q K^T + mask) V with a backward pass.

    q [B,Hq,Tq,D], k and v [B,Hkv,Tkv,D] on one CUDA device, fp16 or bf16,
    Hq a multiple of Hkv (query head h reads KV head h // (Hq // Hkv)).
    ``scale`` defaults to 1/sqrt(D). ``causal`` masks keys after the query
    (top-left aligned); ``window`` W > 0 masks past keys with q - k >= W.
    Non-contiguous inputs are copied to contiguous ones first. With
    ``return_lse`` the natural-log LSE [B,Hq,Tq] (fp32, no gradient) is
    returned beside O.
    """
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    q, k, v = (t.contiguous() for t in (q, k, v))
    o, lse = FlashAttention.apply(q, k, v, float(scale), bool(causal), int(window))
    return (o, lse) if return_lse else o
