"""attention(): the forward and backward passes as one differentiable PyTorch operation.

The forward calls attn_fwd_ex and keeps O and LSE; the backward calls attn_bwd with the
incoming gradient, so autograd reaches the same kernels as the C ABI (argument marshalling
only). Q, K, V are bf16 CUDA tensors [BH, N, d]; the gradients are returned in bf16 like
the inputs (the kernels compute them in fp32). The bias terms take no gradient.
"""
from __future__ import annotations

import math

from . import ATTN_MASK_CAUSAL, ATTN_MASK_NONE, attn_bwd, attn_fwd_ex, bwd_workspace


def _function():
    import torch

    class _Attention(torch.autograd.Function):
        @staticmethod
        def forward(ctx, q, k, v, mode, bias, key_bias, scale):
            BH, Nq, _ = q.shape
            O = torch.empty((BH, Nq, v.shape[2]), dtype=torch.bfloat16, device=q.device)
            LSE = torch.empty((BH, Nq), dtype=torch.float32, device=q.device)
            attn_fwd_ex(q, k, v, mode, bias, key_bias, scale, O, LSE)
            ctx.save_for_backward(q, k, v, O, LSE)
            ctx.mode, ctx.bias, ctx.key_bias, ctx.scale = mode, bias, key_bias, scale
            return O

        @staticmethod
        @torch.autograd.function.once_differentiable
        def backward(ctx, dO):
            q, k, v, O, LSE = ctx.saved_tensors
            dO = dO.to(torch.bfloat16).contiguous()
            dQ = torch.empty(q.shape, dtype=torch.float32, device=q.device)
            dK = torch.empty(k.shape, dtype=torch.float32, device=q.device)
            dV = torch.empty(v.shape, dtype=torch.float32, device=q.device)
            attn_bwd(q, k, v, O, dO, LSE, ctx.mode, ctx.bias, ctx.key_bias, ctx.scale, dQ, dK, dV,
                     bwd_workspace(q.shape[0], q.shape[1], device=q.device))
            return (dQ.to(q.dtype), dK.to(k.dtype), dV.to(v.dtype), None, None, None, None)

    return _Attention


_FN = None


def attention(q, k, v, causal: bool = False, bias=None, key_bias=None, scale: float | None = None):
    """softmax(q k^T * scale + C) v for bf16 CUDA tensors q [BH, Nq, d], k [BH, Nk, d],
    v [BH, Nk, d_v], differentiable in q, k and v. C is the causal mask (aligned at the
    last key) and/or `bias` (fp32 [BH, Nq, Nk], or [Nq, Nk] for one bias shared by every head)
    or `key_bias` (fp32 [BH, Nk]); scale
    defaults to 1 / sqrt(d). Returns O in bf16. The backward pass is first-order only (no
    double backward), and a bias that requires grad is rejected with ValueError."""
    global _FN
    if _FN is None:
        _FN = _function()
    from . import ATTN_BIAS_DENSE, ATTN_BIAS_KEY, ATTN_BIAS_SHARED

    for name, t in (("bias", bias), ("key_bias", key_bias)):
        if t is not None and t.requires_grad:
            raise ValueError(f"attention(): {name} takes no gradient; pass it detached")
    mode = ATTN_MASK_CAUSAL if causal else ATTN_MASK_NONE
    if bias is not None:
        mode |= ATTN_BIAS_DENSE
        if bias.dim() == 2:  # one [Nq, Nk] bias for every head
            mode |= ATTN_BIAS_SHARED
    if key_bias is not None:
        mode |= ATTN_BIAS_KEY
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    return _FN.apply(q.contiguous(), k.contiguous(), v.contiguous(), mode, bias, key_bias, float(scale))
