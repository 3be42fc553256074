"""One device's block calls (ring_attn_block_fwd / ring_attn_block_bwd) through the C ABI against the
float64 oracle's block functions, for every (query shard, key shard) pair, on the tensor-core path
(bf16, head dim 128 and 64) and the CUDA-core path (float32, or shards the tensor-core kernels do not
tile); plus the blocks folded in ring order, which must give full attention."""
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
    (1, 4, 2, 2048, 128, 4, True, "zigzag", torch.bfloat16),
    (1, 2, 1, 2048, 128, 2, True, "contiguous", torch.bfloat16),
    (1, 2, 2, 2048, 128, 4, True, "striped", torch.bfloat16),
    (2, 2, 1, 1536, 128, 3, False, "zigzag", torch.bfloat16),
    (1, 4, 1, 1024, 64, 2, True, "zigzag", torch.bfloat16),
    (1, 2, 1, 768, 128, 3, True, "zigzag", torch.bfloat16),    # chunks of 128: CUDA-core forward, tensor-core backward
    (1, 2, 1, 512, 128, 4, True, "zigzag", torch.float32),     # CUDA-core
    (1, 1, 1, 384, 64, 3, True, "striped", torch.float32),
]


@pytest.fixture(autouse=True)
def _clean_status():
    torch.cuda.set_device(0)
    ra.device_status()
    yield
    assert ra.device_status() == 0, "a bounded wait ran out inside a kernel"


def shard(t, i, n):
    S = t.shape[2] // n
    return t[:, :, i * S:(i + 1) * S].contiguous()


@pytest.mark.parametrize("B,H,Hkv,L,d,n,causal,layout,dtype", CASES)
def test_block_fwd_every_pair_and_the_ring_fold(B, H, Hkv, L, d, n, causal, layout, dtype):
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=dtype, seed=300 + L + n + d)
    S = L // n
    full_o, full_l = oracle.attn_fwd(x["q"], x["k"], x["v"], n, causal, layout)
    for i in range(n):
        q = shard(x["q"], i, n).to(DEV)
        o_run = torch.empty((B, H, S, d), dtype=torch.float32, device=DEV)
        l_run = torch.empty((B, H, S), dtype=torch.float32, device=DEV)
        for r in range(n):
            j = (i - r) % n
            k, v = shard(x["k"], j, n).to(DEV), shard(x["v"], j, n).to(DEV)
            # the block alone (write mode) against the oracle's block
            o_blk = torch.full((B, H, S, d), float("nan"), device=DEV)
            l_blk = torch.full((B, H, S), float("nan"), device=DEV)
            ra.block_fwd(q, k, v, o_blk, l_blk, n, i, j, False, causal, layout)
            ref_o, ref_l = oracle.block_fwd(shard(x["q"], i, n), shard(x["k"], j, n), shard(x["v"], j, n), L, n,
                                            causal, layout, i, j)
            got_l = to_np(l_blk)
            empty = np.isneginf(ref_l)
            assert np.array_equal(np.isneginf(got_l), empty), f"rows without a visible key differ ({i}, {j})"
            assert np.all(to_np(o_blk)[empty] == 0)
            if (~empty).any():
                assert_close(to_np(o_blk)[~empty], ref_o[~empty], dtype, f"o_part ({i},{j})")
                assert_close(got_l[~empty], ref_l[~empty], dtype, f"lse_part ({i},{j})")
            # and folded into the running state in ring order (the first block writes: o_run starts as NaN)
            if r == 0:
                o_run.fill_(float("nan"))
            ra.block_fwd(q, k, v, o_run, l_run, n, i, j, r > 0, causal, layout)
        out = ra.f32_convert(o_run, dtype)
        assert_close(to_np(out), full_o[:, :, i * S:(i + 1) * S], dtype, f"shard {i} out")
        assert_close(to_np(l_run), full_l[:, :, i * S:(i + 1) * S], dtype, f"shard {i} lse")


@pytest.mark.parametrize("B,H,Hkv,L,d,n,causal,layout,dtype", CASES)
def test_block_bwd_every_pair_both_modes(B, H, Hkv, L, d, n, causal, layout, dtype):
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=dtype, seed=400 + L + n + d, with_dout=True)
    S = L // n
    out, lse = oracle.attn_fwd(x["q"], x["k"], x["v"], n, causal, layout)
    D = (x["dout"].double().numpy() * out).sum(-1)
    # the GPU gets the oracle's lse and D rounded to float32; the oracle's block reads the same values
    lse32, D32 = lse.astype(np.float32), D.astype(np.float32)
    rq, rk, rv = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], n, causal, layout)
    # accumulate mode: per key shard, running dK / dV sums over the query shards
    dk_acc = [ra.f32_zero(torch.empty((B, Hkv, S, d), dtype=torch.float32, device=DEV)) for _ in range(n)]
    dv_acc = [ra.f32_zero(torch.empty((B, Hkv, S, d), dtype=torch.float32, device=DEV)) for _ in range(n)]
    for i in range(n):
        sl = slice(i * S, (i + 1) * S)
        q, do = shard(x["q"], i, n).to(DEV), shard(x["dout"], i, n).to(DEV)
        l_i = torch.from_numpy(np.ascontiguousarray(lse32[:, :, sl])).to(DEV)
        D_i = torch.from_numpy(np.ascontiguousarray(D32[:, :, sl])).to(DEV)
        dq_acc = ra.f32_zero(torch.empty((B, H, S, d), dtype=torch.float32, device=DEV))
        for r in range(n):
            j = (i - r) % n
            k, v = shard(x["k"], j, n).to(DEV), shard(x["v"], j, n).to(DEV)
            # store mode into NaN-filled buffers: every key row is written (zeros where it meets no query)
            dk = torch.full((B, Hkv, S, d), float("nan"), device=DEV)
            dv = torch.full((B, Hkv, S, d), float("nan"), device=DEV)
            dq_blk = ra.f32_zero(torch.empty((B, H, S, d), dtype=torch.float32, device=DEV))
            ra.block_bwd(q, k, v, do, l_i, D_i, dq_blk, dk, dv, n, i, j, False, causal, layout)
            a, b, c = oracle.block_bwd(shard(x["q"], i, n), shard(x["k"], j, n), shard(x["v"], j, n),
                                       shard(x["dout"], i, n), lse32[:, :, sl].astype(np.float64),
                                       D32[:, :, sl].astype(np.float64), L, n, causal, layout, i, j)
            for got, ref, what in ((dq_blk, a, "dq"), (dk, b, "dk"), (dv, c, "dv")):
                g = to_np(got)
                assert np.isfinite(g).all(), f"{what} ({i},{j}) not fully written"
                if np.abs(ref).max() == 0:
                    assert np.abs(g).max() == 0, f"{what} ({i},{j}) should be zero"
                else:
                    assert_close(g, ref, dtype, f"{what} part ({i},{j})")
            ra.block_bwd(q, k, v, do, l_i, D_i, dq_acc, dk_acc[j], dv_acc[j], n, i, j, True, causal, layout)
        assert_close(to_np(dq_acc), rq[:, :, sl], dtype, f"shard {i} dq (all blocks)")
    assert_close(to_np(torch.cat(dk_acc, dim=2)), rk, dtype, "dk (all blocks)")
    assert_close(to_np(torch.cat(dv_acc, dim=2)), rv, dtype, "dv (all blocks)")


@pytest.mark.parametrize("rows,d,dtype", [(1, 128, torch.bfloat16), (13, 128, torch.bfloat16),
                                          (1000, 64, torch.bfloat16), (4099, 128, torch.bfloat16),
                                          (37, 96, torch.bfloat16), (50, 128, torch.float32)])
def test_bwd_preprocess_row_sums(rows, d, dtype):
    """D = rowsum(out * dout) for row counts that fill no whole group of rows (the bf16 kernel for head
    dims 64 and 128 works on 8 or 16 rows per warp) and for the general path, against float64 sums
    of the same rounded inputs; rows past the end are not written."""
    g = torch.Generator().manual_seed(rows * 1000 + d)
    o = torch.randn(rows, d, generator=g).to(dtype)
    do = torch.randn(rows, d, generator=g).to(dtype)
    D = torch.full((rows + 64,), float("nan"), device=DEV)
    ra.bwd_preprocess(o.to(DEV), do.to(DEV), D=D[:rows])
    torch.cuda.synchronize()
    ref = (o.double() * do.double()).sum(-1).numpy()
    got = D[:rows].double().cpu().numpy()
    assert np.allclose(got, ref, rtol=1e-5, atol=1e-5 * np.sqrt(d))
    assert torch.isnan(D[rows:]).all()


@pytest.mark.parametrize("rows,d", [(13, 128), (1000, 64), (37, 96)])
def test_bwd_preprocess_with_a_float32_output(rows, d):
    """D = rowsum(out * dout) with out in float32 and dout in bf16 (the unrounded output), against
    float64 sums of the same values."""
    g = torch.Generator().manual_seed(rows * 7 + d)
    o = torch.randn(rows, d, generator=g)
    do = torch.randn(rows, d, generator=g).to(torch.bfloat16)
    D = ra.bwd_preprocess(o.to(DEV), do.to(DEV))
    torch.cuda.synchronize()
    ref = (o.double() * do.double()).sum(-1).numpy()
    assert np.allclose(D.double().cpu().numpy(), ref, rtol=1e-5, atol=1e-5 * np.sqrt(d))
