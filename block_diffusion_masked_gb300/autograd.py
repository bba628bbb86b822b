"""torch.autograd wrappers over the C ABI (the pages' ``diffusion_attn_func``).

``diffusion_attn_func(q, k, v, block_size)`` mirrors the API of "Fast
Diffusion Attention" (section "Try it"): q, k, v are (batch, 2n, heads,
headdim) bf16 tensors ordered [noisy | clean] (k and v may carry fewer
heads, a divisor of q's: grouped-query / multi-query attention, query head h
reading key/value head h // (heads // kv_heads)); the forward saves out and the
log-sum-exp, and the backward recomputes from them (section 4.5 of
"FlashAttention: Exact Attention Without Materialization").
"""

from __future__ import annotations

import torch

from . import binding


class DiffusionAttnFunc(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, block_size):
        q, k, v = (t.contiguous() for t in (q, k, v))
        if k.shape[2] == q.shape[2]:
            out, lse = binding.dfa_forward(q, k, v, block_size)
        else:
            out, lse = binding.dfa_forward_gqa(q, k, v, block_size)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.block_size = block_size
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse = ctx.saved_tensors
        bwd = binding.dfa_backward if k.shape[2] == q.shape[2] else binding.dfa_backward_gqa
        dq, dk, dv = bwd(q, k, v, out, dout.contiguous(), lse, ctx.block_size)
        return dq, dk, dv, None


class CausalAttnFunc(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v):
        q, k, v = (t.contiguous() for t in (q, k, v))
        out, lse = binding.dfa_causal_forward(q, k, v)
        ctx.save_for_backward(q, k, v, out, lse)
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse = ctx.saved_tensors
        dq, dk, dv = binding.dfa_causal_backward(q, k, v, out, dout.contiguous(), lse)
        return dq, dk, dv


class DiffusionAttnVarlenFunc(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, cu_seqlens, block_size):
        q, k, v = (t.contiguous() for t in (q, k, v))
        cu = [int(x) for x in (cu_seqlens.tolist() if isinstance(cu_seqlens, torch.Tensor)
                               else cu_seqlens)]
        out, lse = binding.dfa_forward_varlen(q, k, v, cu, block_size)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.cu = cu
        ctx.block_size = block_size
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse = ctx.saved_tensors
        dq, dk, dv = binding.dfa_backward_varlen(q, k, v, out, dout.contiguous(), lse, ctx.cu,
                                                 ctx.block_size)
        return dq, dk, dv, None, None


def diffusion_attn_varlen_func(q, k, v, cu_seqlens, block_size):
    """Block-diffusion attention on a packed batch (the pages' varlen API).

    q: (rows, heads, headdim), k, v: (rows, kv_heads, headdim) bf16; sample b
    is rows [cu_seqlens[b], cu_seqlens[b+1]), [noisy | clean], even length.
    """
    return DiffusionAttnVarlenFunc.apply(q, k, v, cu_seqlens, block_size)


def diffusion_attn_func(q, k, v, block_size):
    """Attention under the block-diffusion mask; differentiable."""
    return DiffusionAttnFunc.apply(q, k, v, block_size)


def causal_attn_func(q, k, v):
    """Causal attention on (Bc, L, H, d), any Bc; the yardstick kernels."""
    return CausalAttnFunc.apply(q, k, v)
