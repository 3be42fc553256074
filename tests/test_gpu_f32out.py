"""The forward's float32 output and the backward that takes D from it (ring_attn_fwd_f32out,
ring_attn_bwd_f32out), against the ordinary calls and the float64 oracle, on both kernel paths."""
import numpy as np
import pytest
import torch

import oracle
import sequence_sharded_exact_gb300 as ra
from sequence_sharded_exact_gb300 import synth
from parity_util import assert_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"

CASES = [  # B, H, Hkv, L, d, n, causal, layout, dtype
    (1, 4, 2, 2048, 128, 4, True, "zigzag", torch.bfloat16),     # tensor-core kernels
    (1, 4, 1, 2048, 64, 2, True, "striped", torch.bfloat16),
    (2, 2, 2, 1024, 128, 2, False, "contiguous", torch.bfloat16),
    (1, 2, 1, 384, 128, 3, True, "zigzag", torch.bfloat16),      # CUDA-core kernels (chunks of 64)
    (1, 2, 1, 256, 64, 4, True, "striped", torch.float32),
]


@pytest.fixture(autouse=True)
def _clean_status():
    torch.cuda.set_device(0)
    ra.device_status()
    yield
    assert ra.device_status() == 0, "a bounded wait ran out inside a kernel"


@pytest.mark.parametrize("B,H,Hkv,L,d,n,causal,layout,dtype", CASES)
def test_float32_output_rounds_to_the_ordinary_output(B, H, Hkv, L, d, n, causal, layout, dtype):
    """The float32 output, rounded to the inputs' dtype, is the ordinary forward's output bit for bit
    (the same arithmetic, the rounding moved out of the kernel); lse is the same; and it matches the
    oracle."""
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=dtype, seed=301, with_dout=False)
    q, k, v = (x[t].to(DEV) for t in ("q", "k", "v"))
    o32, l32 = ra.fwd_f32out(q, k, v, n, causal, layout)
    o, l = ra.fwd(q, k, v, n, causal, layout)
    torch.cuda.synchronize()
    assert o32.dtype == torch.float32
    assert torch.equal(ra.f32_convert(o32, dtype), o) and torch.equal(l32, l)
    ref_o, ref_l = oracle.attn_fwd(x["q"], x["k"], x["v"], n, causal, layout)
    assert_close(to_np(o32), ref_o, dtype, "out (float32)")


@pytest.mark.parametrize("B,H,Hkv,L,d,n,causal,layout,dtype", CASES)
def test_backward_with_D_from_the_float32_output(B, H, Hkv, L, d, n, causal, layout, dtype):
    """ring_attn_bwd_f32out against the oracle's exact gradient (D from the exact output); for
    float32 inputs it is the ordinary backward."""
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=dtype, seed=302, with_dout=True)
    q, k, v, do = (x[t].to(DEV) for t in ("q", "k", "v", "dout"))
    o32, lse = ra.fwd_f32out(q, k, v, n, causal, layout)
    dq, dk, dv = ra.bwd_f32out(q, k, v, o32, lse, do, n, causal, layout)
    torch.cuda.synchronize()
    rq, rk, rv = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], n, causal, layout)
    for got, ref, name in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        assert_close(to_np(got), ref, dtype, name)
    if dtype == torch.float32:
        o, l = ra.fwd(q, k, v, n, causal, layout)
        gq, gk, gv = ra.bwd(q, k, v, o, l, do, n, causal, layout)
        torch.cuda.synchronize()
        assert torch.equal(gk, dk) and torch.equal(gv, dv)
        assert torch.allclose(gq, dq, rtol=1e-6, atol=1e-6)


def test_autograd_keeps_the_float32_output_for_the_backward():
    B, H, Hkv, L, d, n = 1, 4, 2, 2048, 128, 4
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=torch.bfloat16, seed=303, with_dout=True)
    q, k, v = (x[t].to(DEV).requires_grad_(True) for t in ("q", "k", "v"))
    do = x["dout"].to(DEV)
    out = ra.ring_attention(q, k, v, n, True, "zigzag", f32_out=True)
    (out.float() * do.float()).sum().backward()
    torch.cuda.synchronize()
    o32, lse = ra.fwd_f32out(q.detach(), k.detach(), v.detach(), n, True, "zigzag")
    assert out.dtype == torch.bfloat16 and torch.equal(out.detach(), ra.f32_convert(o32, torch.bfloat16))
    gq, gk, gv = ra.bwd_f32out(q.detach(), k.detach(), v.detach(), o32, lse, do, n, True, "zigzag",
                               grad_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert torch.equal(k.grad, gk) and torch.equal(v.grad, gv)
    assert torch.allclose(q.grad.float(), gq.float(), rtol=2 ** -7, atol=2 ** -7)
