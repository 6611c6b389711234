"""torch.autograd wrapper of one layer of the sparse attention (argument marshalling only).

``fib_attention(plan, layer, q, k, v, alpha)`` returns O; its backward calls the library's
backward, which returns dQ, dK, dV and, in INTERP mode, dl/dalpha of the layer ("Depth-
Staggered Fibonacci Spacing for Sparse Attention", Methodology > "Implementation": the
interpolated rows give alpha a gradient).  ``alpha`` is the per-layer alpha vector on the
device (float32, one entry per layer of the plan); its gradient is nonzero at ``layer`` only.
Every step runs in the CUDA library; nothing here computes attention.  Where the forward
prepares K'/V' rows (bf16, W <= 16), the Function keeps that workspace for the backward in
place of k and v (the same bytes) and the backward starts from it.
"""
import torch

from . import fib_attn as fa


class _FibAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, alpha, plan, layer):
        B, H, N = q.shape[:3]
        need = fa.fib_attn_fwd_workspace_size(plan, B, H, N, q.dtype)
        ctx.plan, ctx.layer, ctx.prepared = plan, layer, need > 0
        if ctx.prepared:
            kv = torch.empty(need, dtype=torch.uint8, device=q.device)
            o, lse = fa.fib_attn_fwd(plan, layer, q, k, v, alpha_dev=alpha, workspace=kv)
            ctx.save_for_backward(q, kv, o, lse, alpha)
        else:
            o, lse = fa.fib_attn_fwd(plan, layer, q, k, v, alpha_dev=alpha)
            ctx.save_for_backward(q, k, v, o, lse, alpha)
        return o

    @staticmethod
    def backward(ctx, dO):
        if ctx.prepared:
            q, kv, o, lse, alpha = ctx.saved_tensors
            dq, dk, dv, da = fa.fib_attn_bwd_prepared(ctx.plan, ctx.layer, q, kv, o, lse, dO.contiguous(),
                                                      alpha_dev=alpha)
        else:
            q, k, v, o, lse, alpha = ctx.saved_tensors
            dq, dk, dv, da = fa.fib_attn_bwd(ctx.plan, ctx.layer, q, k, v, o, lse, dO.contiguous(),
                                             alpha_dev=alpha)
        dalpha = None
        if alpha is not None and ctx.needs_input_grad[3]:
            dalpha = torch.zeros_like(alpha)
            dalpha[ctx.layer] = da[0]
        return dq, dk, dv, dalpha, None, None


def fib_attention(plan, layer: int, q, k, v, alpha=None):
    """O of layer ``layer`` for q, k, v [B, H, N, 64] (contiguous CUDA, float32 or bfloat16);
    ``alpha``: device float32 [n_layers] (INTERP: used and differentiated) or None."""
    return _FibAttention.apply(q, k, v, alpha, plan, layer)
