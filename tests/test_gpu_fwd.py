"""GPU parity of the forward path (through the C ABI) against the float64 oracle."""
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


def inputs(B, H, Hkv, L, d, dtype, seed, spike=0.0, dout=False):
    return synth.make_inputs(B, H, Hkv, L, d, dtype=dtype, seed=seed, spike_frac=spike,
                             with_dout=dout, device="cpu")


def run_fwd_full(B, H, Hkv, L, d, n, causal, layout, dtype, seed, spike=0.0, expect_path=None):
    x = inputs(B, H, Hkv, L, d, dtype, seed, spike)
    if expect_path:
        assert ra.fwd_path(B, H, Hkv, L, d, n, causal, layout, dtype) == expect_path
    q, k, v = (x[t].to(DEV) for t in ("q", "k", "v"))
    out, lse = ra.fwd(q, k, v, n, causal, layout)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attn_fwd(x["q"], x["k"], x["v"], n, causal, layout)
    assert_close(to_np(out), ref_o, dtype, "out")
    assert_close(to_np(lse), ref_l, dtype, "lse")
    return out, lse, x


def test_tiny_f32_workload():
    """The tiny fp32 workload: B1 H1 d64 L256 n4, non-causal, contiguous (max-abs 1e-4)."""
    w = synth.WORKLOADS["tiny_f32"]
    run_fwd_full(w["B"], w["H"], w["Hkv"], w["L"], w["d"], w["n"], w["causal"], w["layout"],
                 w["dtype"], w["seed"], expect_path="simt")


TC_CASES = [
    # B, H, Hkv, L, n, causal, layout
    (1, 2, 2, 512, 1, True, "contiguous"),
    (1, 2, 1, 1024, 2, True, "zigzag"),
    (2, 4, 2, 2048, 4, True, "zigzag"),
    (1, 4, 4, 1024, 4, False, "contiguous"),
    (1, 8, 2, 2048, 2, False, "zigzag"),
    (1, 4, 1, 4096, 8, True, "zigzag"),
    (1, 2, 2, 768, 3, True, "contiguous"),   # odd number of 256-row blocks
    (1, 3, 1, 1280, 1, True, "contiguous"),  # n = 1, odd blocks, GQA 3:1
    (1, 4, 2, 2048, 8, True, "contiguous"),
    (1, 4, 2, 2048, 4, True, "striped"),
    (1, 2, 1, 1024, 2, False, "striped"),
    (2, 2, 2, 3072, 3, True, "striped"),     # 4 blocks of 256 rows per shard
    (1, 4, 1, 4096, 8, True, "striped"),     # 2 blocks per shard: one mirrored pair
]


@pytest.mark.parametrize("B,H,Hkv,L,n,causal,layout", TC_CASES)
def test_tcgen05_fwd_matches_oracle(B, H, Hkv, L, n, causal, layout):
    run_fwd_full(B, H, Hkv, L, 128, n, causal, layout, torch.bfloat16, seed=L + n + H,
                 expect_path="tcgen05")


TC_CASES_D64 = [
    # B, H, Hkv, L, n, causal, layout  (head dim 64: the same kernel with one 64-column box per row)
    (1, 2, 2, 512, 1, True, "contiguous"),
    (2, 4, 2, 2048, 4, True, "zigzag"),
    (1, 8, 2, 2048, 2, False, "zigzag"),
    (1, 3, 1, 1280, 1, True, "contiguous"),
    (1, 4, 2, 2048, 4, True, "striped"),
]


@pytest.mark.parametrize("B,H,Hkv,L,n,causal,layout", TC_CASES_D64)
def test_tcgen05_fwd_head_dim_64_matches_oracle(B, H, Hkv, L, n, causal, layout):
    run_fwd_full(B, H, Hkv, L, 64, n, causal, layout, torch.bfloat16, seed=L + n + H + 64,
                 expect_path="tcgen05")


def test_tcgen05_fwd_head_dim_64_steps_and_host_buffers():
    """Head dim 64 through the ring-step forms and the host-buffer forward: the same results as
    the fused call (step folds: within the bf16 bound of the oracle; host buffers: identical)."""
    B, H, Hkv, L, d, n = 1, 4, 2, 2048, 64, 4
    x = inputs(B, H, Hkv, L, d, torch.bfloat16, seed=71)
    q, k, v = (x[t].to(DEV) for t in ("q", "k", "v"))
    out_f, lse_f = ra.fwd(q, k, v, n, True, "zigzag")
    out_s, lse_s = ra.fwd_stepwise(q, k, v, n, True, "zigzag")
    out_h, lse_h = ra.fwd_host(*(x[t].pin_memory() for t in ("q", "k", "v")), n, True, "zigzag")
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attn_fwd(x["q"], x["k"], x["v"], n, True, "zigzag")
    assert_close(to_np(out_s), ref_o, torch.bfloat16, "stepwise out")
    assert_close(to_np(lse_s), ref_l, torch.bfloat16, "stepwise lse")
    assert torch.equal(out_h, out_f.cpu()) and torch.equal(lse_h, lse_f.cpu())


def test_tcgen05_fwd_large_keys():
    """1% of key rows scaled x8: the running maximum jumps late in the walk."""
    run_fwd_full(1, 4, 2, 2048, 128, 4, True, "zigzag", torch.bfloat16, seed=5, spike=0.01,
                 expect_path="tcgen05")


SIMT_CASES = [
    # B, H, Hkv, L, d, n, causal, layout, dtype
    (1, 2, 1, 1000, 128, 5, True, "contiguous", torch.bfloat16),   # ragged: S = 200
    (1, 2, 2, 384, 128, 3, True, "zigzag", torch.bfloat16),        # chunks of 64
    (1, 2, 2, 512, 64, 2, True, "zigzag", torch.bfloat16),         # head dim 64
    (2, 4, 2, 640, 128, 5, True, "zigzag", torch.float32),
    (1, 2, 1, 300, 64, 3, False, "contiguous", torch.float32),
    (1, 2, 2, 384, 128, 3, True, "striped", torch.bfloat16),       # S = 128: below a block
    (1, 2, 1, 600, 64, 5, True, "striped", torch.float32),
    # degenerate shards: one row per shard / per zigzag chunk
    (1, 2, 1, 4, 64, 4, True, "contiguous", torch.float32),
    (1, 2, 2, 8, 128, 4, True, "zigzag", torch.bfloat16),
    (2, 1, 1, 6, 64, 3, True, "striped", torch.float32),
    (1, 1, 1, 1, 64, 1, True, "contiguous", torch.float32),        # a single token
]


@pytest.mark.parametrize("B,H,Hkv,L,d,n,causal,layout,dtype", SIMT_CASES)
def test_simt_fwd_matches_oracle(B, H, Hkv, L, d, n, causal, layout, dtype):
    run_fwd_full(B, H, Hkv, L, d, n, causal, layout, dtype, seed=L + d, expect_path="simt")


@pytest.mark.parametrize("B,H,Hkv,L,d,n,layout,dtype", [
    (1, 4, 2, 1024, 128, 4, "zigzag", torch.bfloat16),       # tensor-core ring steps
    (1, 2, 2, 1024, 128, 2, "contiguous", torch.bfloat16),
    (1, 2, 1, 600, 64, 3, "zigzag", torch.float32),          # SIMT ring steps
    (1, 4, 2, 2048, 128, 4, "striped", torch.bfloat16),
    (1, 2, 1, 600, 64, 3, "striped", torch.float32),
])
def test_stepwise_ring_matches_oracle_and_fused(B, H, Hkv, L, d, n, layout, dtype):
    """n ring-step launches, each folded into the running result in its epilogue, equal full
    attention and the fused kernel."""
    x = inputs(B, H, Hkv, L, d, dtype, seed=77)
    q, k, v = (x[t].to(DEV) for t in ("q", "k", "v"))
    out_s, lse_s = ra.fwd_stepwise(q, k, v, n, True, layout)
    out_f, lse_f = ra.fwd(q, k, v, n, True, layout)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attn_fwd(x["q"], x["k"], x["v"], n, True, layout)
    assert_close(to_np(out_s), ref_o, dtype, "stepwise out")
    assert_close(to_np(lse_s), ref_l, dtype, "stepwise lse")
    assert_close(to_np(out_s), to_np(out_f), dtype, "stepwise vs fused")


@pytest.mark.parametrize("B,H,Hkv,L,d,n,layout,dtype", [
    (1, 4, 2, 1024, 128, 4, "zigzag", torch.bfloat16),       # tensor-core ring steps
    (2, 2, 1, 768, 128, 3, "striped", torch.bfloat16),
    (1, 2, 1, 600, 64, 3, "contiguous", torch.float32),      # CUDA-core ring steps
])
def test_stepwise_non_causal_matches_oracle(B, H, Hkv, L, d, n, layout, dtype):
    """Without the causal mask every ring step sees the whole K/V shard: the folded steps equal full
    (unmasked) attention."""
    x = inputs(B, H, Hkv, L, d, dtype, seed=81)
    q, k, v = (x[t].to(DEV) for t in ("q", "k", "v"))
    out_s, lse_s = ra.fwd_stepwise(q, k, v, n, False, layout)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attn_fwd(x["q"], x["k"], x["v"], n, False, layout)
    assert_close(to_np(out_s), ref_o, dtype, "stepwise out")
    assert_close(to_np(lse_s), ref_l, dtype, "stepwise lse")


@pytest.mark.parametrize("B,H,Hkv,L,d,n,layout,dtype", [
    (1, 4, 2, 1024, 128, 4, "zigzag", torch.bfloat16),
    (1, 2, 1, 600, 64, 3, "striped", torch.float32),
])
def test_ring_steps_with_lse_merge_match_oracle(B, H, Hkv, L, d, n, layout, dtype):
    """n separate ring-step partials folded by the LSE merge kernel equal full attention (the
    two-kernel form of the step loop)."""
    x = inputs(B, H, Hkv, L, d, dtype, seed=78)
    q, k, v = (x[t].to(DEV) for t in ("q", "k", "v"))
    o_acc, l_acc = ra.ring_step_fwd(q, k, v, n, 0, True, layout)
    for step in range(1, n):
        o, lse = ra.ring_step_fwd(q, k, v, n, step, True, layout)
        ra.lse_merge(o_acc, l_acc, o, lse)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attn_fwd(x["q"], x["k"], x["v"], n, True, layout)
    assert_close(o_acc.cpu().numpy(), ref_o, dtype, "merged out")
    assert_close(l_acc.cpu().numpy(), ref_l, dtype, "merged lse")


@pytest.mark.parametrize("L,d,n,layout,dtype", [
    (1024, 128, 4, "zigzag", torch.bfloat16),      # tensor-core epilogue
    (2048, 128, 4, "striped", torch.bfloat16),
    (1024, 128, 4, "contiguous", torch.bfloat16),  # rows that see nothing at a step
    (600, 64, 3, "zigzag", torch.float32),         # CUDA-core epilogue
    (400, 64, 4, "contiguous", torch.float32),
])
def test_ring_step_accumulate_equals_step_then_merge(L, d, n, layout, dtype):
    """Folding a ring step into an arbitrary running state inside the kernel equals computing the
    step's partial and merging it with the LSE merge: from a random state (finite rows, empty
    rows with lse = -inf, rows with large lse gaps either way), at every step."""
    B, H, Hkv = 1, 4, 2
    x = inputs(B, H, Hkv, L, d, dtype, seed=79)
    q, k, v = (x[t].to(DEV) for t in ("q", "k", "v"))
    g = torch.Generator().manual_seed(80)
    o0 = torch.randn(B, H, L, d, generator=g)
    l0 = torch.randn(B, H, L, generator=g) * 4
    l0[..., ::5] = float("-inf")
    l0[..., 1::13] += 40.0
    l0[..., 2::13] -= 40.0
    for step in range(n):
        o_ref, l_ref = o0.clone().to(DEV), l0.clone().to(DEV)
        o, lse = ra.ring_step_fwd(q, k, v, n, step, True, layout)
        ra.lse_merge(o_ref, l_ref, o, lse)
        o_acc, l_acc = o0.clone().to(DEV), l0.clone().to(DEV)
        ra.ring_step_fwd_accumulate(q, k, v, n, step, o_acc, l_acc, True, layout)
        torch.cuda.synchronize()
        seen = torch.isfinite(l_ref.cpu())  # rows empty before and after hold no defined output
        assert torch.equal(torch.isneginf(l_acc.cpu()), torch.isneginf(l_ref.cpu())), step
        dl = (l_acc.cpu() - l_ref.cpu())[seen].abs().max().item()
        do = (o_acc.cpu() - o_ref.cpu())[seen].abs().max().item()
        assert dl <= 1e-5 and do <= 2e-5, (step, dl, do)


@pytest.mark.parametrize("d,L,dtype", [(128, 1024, torch.bfloat16), (64, 400, torch.float32)])
def test_ring_step_skips_future_shards(d, L, dtype):
    """Contiguous causal: at step r the shards i < r face a later shard and see nothing
    (o = 0, lse = -inf); every other shard gets its block's attention."""
    n = 4
    S = L // n
    x = inputs(1, 2, 1, L, d, dtype, seed=3)
    q, k, v = (x[t].to(DEV) for t in ("q", "k", "v"))
    for step in range(n):
        o, lse = ra.ring_step_fwd(q, k, v, n, step, True, "contiguous")
        torch.cuda.synchronize()
        lse_np = lse.cpu().numpy()
        for i in range(n):
            rows = slice(i * S, (i + 1) * S)
            if i < step:
                assert np.all(np.isneginf(lse_np[:, :, rows]))
                assert torch.count_nonzero(o[:, :, rows]).item() == 0
            else:
                assert np.all(np.isfinite(lse_np[:, :, rows]))


def test_constant_v_gives_constant_output():
    x = inputs(1, 4, 2, 1024, 128, torch.bfloat16, seed=9)
    c = torch.randn(128, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    v = c.expand(1, 2, 1024, 128).contiguous().to(DEV)
    out, _ = ra.fwd(x["q"].to(DEV), x["k"].to(DEV), v, 4, True, "zigzag")
    torch.cuda.synchronize()
    err = (out.float().cpu() - c.float()).abs().max().item()
    assert err <= 2e-2 * max(1.0, c.float().abs().max().item())


@pytest.mark.parametrize("rows,d", [(1000, 128), (999, 128), (1, 128), (333, 64)])
def test_lse_merge_kernel(rows, d):
    """Merging two partials of a row set equals the log-sum-exp combination of their weights."""
    g = torch.Generator().manual_seed(4)
    oa, ob = torch.randn(rows, d, generator=g), torch.randn(rows, d, generator=g)
    la, lb = torch.randn(rows, generator=g) * 5, torch.randn(rows, generator=g) * 5
    lb[::7] = float("-inf")   # empty partials leave the row unchanged
    la[::11] = float("-inf")  # empty accumulators take the partial
    la[::77] = float("-inf")
    o_acc, l_acc = oa.clone().to(DEV), la.clone().to(DEV)
    ra.lse_merge(o_acc, l_acc, ob.to(DEV), lb.to(DEV))
    torch.cuda.synchronize()
    a64, b64 = la.double(), lb.double()
    lse = torch.logaddexp(a64, b64)
    wa = torch.where(torch.isneginf(a64), 0.0, torch.exp(a64 - lse))
    wb = torch.where(torch.isneginf(b64), 0.0, torch.exp(b64 - lse))
    oa64 = torch.where(torch.isneginf(a64)[:, None], 0.0, oa.double())
    ref_o = wa[:, None] * oa64 + wb[:, None] * ob.double()
    got_o = o_acc.cpu().double()
    both_empty = torch.isneginf(a64) & torch.isneginf(b64)
    ref_o[both_empty] = got_o[both_empty]
    assert torch.allclose(l_acc.cpu().double(), lse, atol=1e-5, rtol=0, equal_nan=False)
    assert (got_o - ref_o).abs().max().item() < 1e-5


@pytest.mark.parametrize("d,L,dtype", [(128, 2048, torch.bfloat16), (64, 600, torch.float32)])
def test_striped_ring_step_first_rows(d, L, dtype):
    """Striped causal: at step r > 0 the query shard i faces key shard j = i - r (mod n).  Where
    j > i the shard's first query row (natural position i) sees none of shard j (o = 0,
    lse = -inf); every other row sees at least shard j's first key."""
    n = 4
    S = L // n
    x = inputs(1, 2, 1, L, d, dtype, seed=8)
    q, k, v = (x[t].to(DEV) for t in ("q", "k", "v"))
    for step in range(1, n):
        o, lse = ra.ring_step_fwd(q, k, v, n, step, True, "striped")
        torch.cuda.synchronize()
        lse_np = lse.cpu().numpy()
        for i in range(n):
            j = (i - step) % n
            rows = lse_np[:, :, i * S:(i + 1) * S]
            assert np.all(np.isfinite(rows[:, :, 1:]))
            if j > i:
                assert np.all(np.isneginf(rows[:, :, 0]))
                assert torch.count_nonzero(o[:, :, i * S]).item() == 0
            else:
                assert np.all(np.isfinite(rows[:, :, 0]))


@pytest.mark.parametrize("B,H,Hkv,L,d,n,layout,dtype,pinned", [
    (2, 4, 2, 2048, 128, 4, "zigzag", torch.bfloat16, True),   # tensor-core groups
    (1, 2, 1, 600, 64, 3, "striped", torch.float32, True),     # CUDA-core groups
    (1, 4, 4, 1024, 128, 2, "contiguous", torch.bfloat16, False),
    (2, 8, 4, 2048, 128, 4, "striped", torch.bfloat16, True),   # 8 groups over 2 slots, 2 streams
])
def test_fwd_host_equals_device_forward(B, H, Hkv, L, d, n, layout, dtype, pinned):
    """ring_attn_fwd_host (host buffers, per-group copies overlapped with compute) returns exactly
    what ring_attn_fwd returns on device-resident inputs (same kernels, no atomics)."""
    x = inputs(B, H, Hkv, L, d, dtype, seed=L + 17)
    hq, hk, hv = (x[t].pin_memory() if pinned else x[t].clone() for t in ("q", "k", "v"))
    out_h, lse_h = ra.fwd_host(hq, hk, hv, n, True, layout)
    torch.cuda.current_stream().synchronize()
    out_d, lse_d = ra.fwd(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), n, True, layout)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(lse_h, lse_d.cpu())
    ref_o, ref_l = oracle.attn_fwd(x["q"], x["k"], x["v"], n, True, layout)
    assert_close(to_np(out_h), ref_o, dtype, "out")


def test_fwd_host_back_to_back_calls_share_a_workspace():
    """Two host-buffer forwards enqueued back to back on one stream with one workspace (no sync in
    between): the second call's copies and kernels wait for the first call's, so each returns the
    device forward of its own inputs."""
    B, H, Hkv, L, d, n = 1, 8, 4, 2048, 128, 4
    xa = inputs(B, H, Hkv, L, d, torch.bfloat16, seed=91)
    xb = inputs(B, H, Hkv, L, d, torch.bfloat16, seed=92)
    ha = [xa[t].pin_memory() for t in ("q", "k", "v")]
    hb = [xb[t].pin_memory() for t in ("q", "k", "v")]
    need = ra.library().ring_attn_fwd_host_workspace_size(H, Hkv, L, d, 1)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    out_a, lse_a = ra.fwd_host(*ha, n, True, "zigzag", workspace=ws)
    out_b, lse_b = ra.fwd_host(*hb, n, True, "zigzag", workspace=ws)
    torch.cuda.current_stream().synchronize()
    for x, o, l in ((xa, out_a, lse_a), (xb, out_b, lse_b)):
        od, ld = ra.fwd(x["q"].to(DEV), x["k"].to(DEV), x["v"].to(DEV), n, True, "zigzag")
        torch.cuda.synchronize()
        assert torch.equal(o, od.cpu()) and torch.equal(l, ld.cpu())
