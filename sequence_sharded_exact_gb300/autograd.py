"""Ring attention as a differentiable PyTorch operation.

``ring_attention`` runs the library's forward and, when a gradient is needed, its backward: the
same ``ring_attn_fwd`` / ``ring_attn_bwd`` entry points as ``fwd`` and ``bwd`` in the binding.  The
forward saves its output and log-sum-exp; the backward recomputes the attention weights from them
(nothing quadratic is stored).  Gradients come back in the dtype of the inputs.

With ``f32_out=True`` (bf16 inputs) the forward keeps its output in float32 for the backward
(``ring_attn_fwd_f32out``, then ``ring_attn_f32_convert`` for the returned bf16 output) and the
backward takes D = rowsum(dout * out) from it (``ring_attn_bwd_f32out``) instead of from the rounded
output: twice the saved output's memory, and gradients closer to the exact ones where a gradient is
a short sum of large, cancelling terms (the first positions of a causal sequence).
"""
import torch

from . import binding


class _RingAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, n_shards, causal, layout, f32_out):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        f32_out = bool(f32_out) and q.dtype != torch.float32
        if f32_out:
            saved, lse = binding.fwd_f32out(q, k, v, n_shards, causal, layout)
            out = binding.f32_convert(saved, q.dtype)
        else:
            out, lse = binding.fwd(q, k, v, n_shards, causal, layout)
            saved = out
        ctx.save_for_backward(q, k, v, saved, lse)
        ctx.cfg = (n_shards, causal, layout, f32_out)
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, saved, lse = ctx.saved_tensors
        n_shards, causal, layout, f32_out = ctx.cfg
        call = binding.bwd_f32out if f32_out else binding.bwd
        dq, dk, dv = call(q, k, v, saved, lse, dout.contiguous(), n_shards, causal, layout, grad_dtype=q.dtype)
        return dq, dk, dv, None, None, None, None


def ring_attention(q, k, v, n_shards, causal=True, layout="zigzag", f32_out=False):
    """Exact attention of q [B,H,L,d] over k, v [B,Hkv,L,d] (sequence axis in the layout's order),
    computed as the ring over n_shards shards; differentiable with respect to q, k and v.
    f32_out: keep the forward's output in float32 for the backward's D (see the module notes)."""
    return _RingAttention.apply(q, k, v, n_shards, causal, layout, f32_out)
