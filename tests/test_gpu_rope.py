"""GPU parity of ring_attn_rope (rotary positions by natural position) against the float64 oracle,
alone, in front of the ring forward, and in the gradient chain of the ring backward."""
import numpy as np
import pytest
import torch

import oracle
import sequence_sharded_exact_gb300 as ra
from sequence_sharded_exact_gb300 import synth
from parity_util import assert_close, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _clean_status():
    torch.cuda.set_device(0)
    ra.device_status()
    yield
    assert ra.device_status() == 0, "a bounded wait ran out inside a kernel"


CASES = [
    # B, H, L, d, n, layout, dtype, base, inverse
    (1, 2, 1000, 64, 5, "contiguous", torch.float32, 10000.0, False),  # ragged: S = 200
    (2, 3, 768, 128, 3, "zigzag", torch.bfloat16, 10000.0, False),
    (1, 4, 1024, 128, 4, "striped", torch.float32, 500000.0, False),
    (1, 2, 512, 128, 2, "zigzag", torch.float32, 10000.0, True),
    (1, 1, 131072, 128, 8, "zigzag", torch.float32, 10000.0, False),  # positions up to 131071
]


@pytest.mark.parametrize("B,H,L,d,n,layout,dtype,base,inverse", CASES)
def test_rope_matches_oracle(B, H, L, d, n, layout, dtype, base, inverse):
    x = torch.randn(B, H, L, d, generator=torch.Generator().manual_seed(L + d)).to(dtype)
    ref = oracle.rope(x, n, layout, base=base, inverse=inverse)
    got = ra.rope(x.to(DEV), n, layout, base=base, inverse=inverse)
    torch.cuda.synchronize()
    assert_close(to_np(got), ref, dtype, "rope", stored_bf16=dtype == torch.bfloat16)


def test_rope_inverse_undoes_rope():
    x = torch.randn(1, 4, 4096, 128, generator=torch.Generator().manual_seed(3)).to(DEV)
    y = ra.rope(x.clone(), 8, "zigzag")
    z = ra.rope(y.clone(), 8, "zigzag", inverse=True)
    torch.cuda.synchronize()
    assert (z - x).abs().max().item() < 2e-6
    assert (y - x).abs().max().item() > 0.1


def test_rope_then_ring_forward_matches_oracle():
    """Positions follow the rows: rotating q and k by natural position, then the ring forward on the
    sharded buffers, equals exact attention of the rotated sequence."""
    B, H, Hkv, L, d, n, layout = 1, 4, 2, 2048, 128, 4, "zigzag"
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=torch.bfloat16, seed=41)
    q, k, v = (x[t].to(DEV) for t in ("q", "k", "v"))
    ra.rope(q, n, layout)
    ra.rope(k, n, layout)
    out, lse = ra.fwd(q, k, v, n, True, layout)
    torch.cuda.synchronize()
    # the oracle reads the same bf16 rotated values the kernels read
    ref_o, ref_l = oracle.attn_fwd(q.cpu(), k.cpu(), x["v"], n, True, layout)
    assert_close(to_np(out), ref_o, torch.bfloat16, "out")
    assert_close(to_np(lse), ref_l, torch.bfloat16, "lse")
    # and those rotated values are the oracle's rotation of the inputs (bf16-stored)
    assert_close(to_np(q), oracle.rope(x["q"], n, layout), torch.bfloat16, "rotated q", stored_bf16=True)


@pytest.mark.parametrize("layout", ["zigzag", "striped"])
def test_rope_gradient_chain(layout):
    """ring backward at the rotated inputs, then the inverse rotation of dq and dk (float32), against
    the oracle's chain."""
    B, H, Hkv, L, d, n = 1, 2, 1, 1024, 128, 4
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=torch.bfloat16, seed=43, with_dout=True)
    q, k, v, do = (x[t].to(DEV) for t in ("q", "k", "v", "dout"))
    ra.rope(q, n, layout)
    ra.rope(k, n, layout)
    out, lse = ra.fwd(q, k, v, n, True, layout)
    dq, dk, dv = ra.bwd(q, k, v, out, lse, do, n, True, layout)
    ra.rope(dq, n, layout, inverse=True)
    ra.rope(dk, n, layout, inverse=True)
    torch.cuda.synchronize()
    rq, rk, rv = oracle.attn_bwd(q.cpu(), k.cpu(), x["v"], x["dout"], n, True, layout)
    assert_close(to_np(dq), oracle.rope(rq.astype(np.float32), n, layout, inverse=True), torch.bfloat16, "dq")
    assert_close(to_np(dk), oracle.rope(rk.astype(np.float32), n, layout, inverse=True), torch.bfloat16, "dk")
    assert_close(to_np(dv), rv, torch.bfloat16, "dv")


@pytest.mark.parametrize("layout,n", [("contiguous", 4), ("zigzag", 4), ("striped", 8), ("zigzag", 1)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("inverse", [False, True])
def test_block_rope_equals_the_whole_sequence_rotation(layout, n, dtype, inverse):
    """One device's rotation of its own shard (ring_attn_block_rope) gives bit for bit the rows of the
    whole-sequence rotation: every row turns by its natural position, wherever it is stored."""
    B, H, L, d = 2, 3, 4096, 128
    x = synth.make_inputs(B, H, H, L, d, dtype=dtype, seed=77, device="cuda:0")["q"]
    whole = ra.rope(x.clone(), n, layout, base=500000.0, inverse=inverse)
    S = L // n
    for i in range(n):
        part = x[:, :, i * S:(i + 1) * S].contiguous()
        ra.block_rope(part, n, i, layout, base=500000.0, inverse=inverse)
        assert torch.equal(part, whole[:, :, i * S:(i + 1) * S]), f"shard {i}"
