"""apply_rotary_emb for training: torch autograd over libastr's RoPE kernels.

AstrAI internals, "Rotary Position Embedding (RoPE)", and inference guide, "Rotary Embedding
Backend": training applies RoPE as a complex multiply that autograd differentiates. Here the
forward rotates q and k with ``astr_rope_apply`` (no cache write) and the backward applies the
transposed rotation with ``astr_rope_backward``, so both passes run in the library's kernels;
this module only reshapes tensors and allocates the outputs.
"""
from __future__ import annotations

import torch

from . import astr_rope_apply, astr_rope_backward


def _flat(x):
    # [..., heads, head_dim] -> [tokens, heads, head_dim]
    return x.contiguous().view(-1, x.shape[-2], x.shape[-1])


class RotaryApply(torch.autograd.Function):
    """(q, k) -> (R q, R k) per token position; the gradient is (R^T dq, R^T dk)."""

    @staticmethod
    def forward(ctx, q, k, freqs_cis, position_ids):
        pos = position_ids.reshape(-1).to(torch.int32).contiguous()
        qf, kf = _flat(q), _flat(k)
        if qf.shape[0] != pos.numel() or kf.shape[0] != pos.numel():
            raise ValueError("q, k and position_ids must cover the same tokens")
        q_out, k_out = torch.empty_like(qf), torch.empty_like(kf)
        astr_rope_apply(qf, q_out, kf, k_out, freqs_cis, pos)
        ctx.save_for_backward(freqs_cis, pos)
        return q_out.view(q.shape), k_out.view(k.shape)

    @staticmethod
    def backward(ctx, grad_q_out, grad_k_out):
        freqs_cis, pos = ctx.saved_tensors
        gq, gk = _flat(grad_q_out), _flat(grad_k_out)
        grad_q, grad_k = torch.empty_like(gq), torch.empty_like(gk)
        astr_rope_backward(gq, grad_q, gk, grad_k, freqs_cis, pos)
        return grad_q.view(grad_q_out.shape), grad_k.view(grad_k_out.shape), None, None


def apply_rotary_emb(q, k, freqs_cis, position_ids):
    """Rotate q [..., n_heads, head_dim] and k [..., n_kv_heads, head_dim] by the positions in
    position_ids (one per token of the leading dimensions), differentiably."""
    return RotaryApply.apply(q, k, freqs_cis, position_ids)
