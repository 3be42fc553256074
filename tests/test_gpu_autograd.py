"""ring_attention as a differentiable PyTorch operation: the gradients autograd produces are the
library backward's, and match the oracle."""
import pytest
import torch

import oracle
import sequence_sharded_exact_gb300 as ra
from sequence_sharded_exact_gb300 import synth
from parity_util import assert_close, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.mark.parametrize("B,H,Hkv,L,d,n,causal,layout,dtype", [
    (1, 4, 2, 1024, 128, 4, True, "zigzag", torch.bfloat16),   # tensor-core path, bf16 gradients
    (1, 2, 1, 384, 64, 3, True, "striped", torch.float32),     # CUDA-core path, fp32 gradients
])
def test_autograd_gradients_are_the_library_backward(B, H, Hkv, L, d, n, causal, layout, dtype):
    torch.cuda.set_device(0)
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=dtype, seed=61, with_dout=True)
    q, k, v = (x[t].to(DEV).requires_grad_(True) for t in ("q", "k", "v"))
    do = x["dout"].to(DEV)
    out = ra.ring_attention(q, k, v, n, causal, layout)
    (out.float() * do.float()).sum().backward()
    torch.cuda.synchronize()
    out_d, lse_d = ra.fwd(q.detach(), k.detach(), v.detach(), n, causal, layout)
    dq, dk, dv = ra.bwd(q.detach(), k.detach(), v.detach(), out_d, lse_d, do, n, causal, layout,
                        grad_dtype=dtype)
    torch.cuda.synchronize()
    assert torch.equal(out.detach(), out_d)
    for got, ref in ((q.grad, dq), (k.grad, dk), (v.grad, dv)):
        assert got.dtype == dtype and got.shape == ref.shape
        # the same kernels; dQ's float atomics may add in another order, which can move a bf16
        # gradient by one unit in its last place
        tol = 1e-5 if dtype == torch.float32 else 2 ** -7
        assert torch.allclose(got.float(), ref.float(), rtol=tol, atol=tol)
    rq, rk, rv = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], n, causal, layout)
    for got, ref, name in ((q.grad, rq, "dq"), (k.grad, rk, "dk"), (v.grad, rv, "dv")):
        assert_close(to_np(got), ref, dtype, name, stored_bf16=dtype == torch.bfloat16)
