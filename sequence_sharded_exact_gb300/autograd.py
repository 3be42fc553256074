"""Ring attention as a differentiable PyTorch operation.

``ring_attention`` runs the library's forward and, when a gradient is needed, its backward: the
same ``ring_attn_fwd`` / ``ring_attn_bwd`` entry points as ``fwd`` and ``bwd`` in the binding.  The
forward saves its output and log-sum-exp; the backward recomputes the attention weights from them
(nothing quadratic is stored).  Gradients come back in the dtype of the inputs.
"""
import torch

from . import binding


class _RingAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, n_shards, causal, layout):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        out, lse = binding.fwd(q, k, v, n_shards, causal, layout)
        ctx.save_for_backward(q, k, v, out, lse)
        ctx.cfg = (n_shards, causal, layout)
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, out, lse = ctx.saved_tensors
        n_shards, causal, layout = ctx.cfg
        dq, dk, dv = binding.bwd(q, k, v, out, lse, dout.contiguous(), n_shards, causal, layout,
                                 grad_dtype=q.dtype)
        return dq, dk, dv, None, None, None


def ring_attention(q, k, v, n_shards, causal=True, layout="zigzag"):
    """Exact attention of q [B,H,L,d] over k, v [B,Hkv,L,d] (sequence axis in the layout's order),
    computed as the ring over n_shards shards; differentiable with respect to q, k and v."""
    return _RingAttention.apply(q, k, v, n_shards, causal, layout)
