"""A seeded sweep of random problem shapes through the C ABI against the float64 oracle: batch, query
and kv heads (GQA ratios 1-4), sequence length, shard count, head dim, layout, causality and dtype
drawn at random (fixed seeds, so the sweep is the same on every run), each checked element by
element -- the fused forward and backward on whichever kernel path the shape takes, and one random
(query shard, key shard) pair of the per-device block calls."""
import numpy as np
import pytest
import torch

import oracle
import sequence_sharded_exact_gb300 as ra
from sequence_sharded_exact_gb300 import synth
from parity_util import assert_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def draw(seed):
    rng = np.random.default_rng(seed)
    layout = ["contiguous", "zigzag", "striped"][rng.integers(3)]
    n = int(rng.choice([1, 2, 3, 4, 8]))
    d = int(rng.choice([64, 128]))
    dtype = torch.bfloat16 if rng.random() < 0.75 else torch.float32
    Hkv = int(rng.integers(1, 3))
    H = Hkv * int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 3))
    unit = 2 * n if layout == "zigzag" else n
    # lengths that land on the tensor-core path (shards or chunks of 256 rows) or off it
    per = int(rng.choice([128, 256, 384, 512])) if dtype == torch.bfloat16 else int(rng.choice([16, 32, 48]))
    L = unit * per
    causal = bool(rng.random() < 0.8)
    return B, H, Hkv, L, d, n, causal, layout, dtype


SEEDS = list(range(9000, 9024))


@pytest.fixture(autouse=True)
def _clean_status():
    torch.cuda.set_device(0)
    ra.device_status()
    yield
    assert ra.device_status() == 0, "a bounded wait ran out inside a kernel"


@pytest.mark.parametrize("seed", SEEDS)
def test_random_shape_forward_backward_and_a_block(seed):
    B, H, Hkv, L, d, n, causal, layout, dtype = draw(seed)
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=dtype, seed=seed, with_dout=True)
    q, k, v, do = (x[t].to(DEV) for t in ("q", "k", "v", "dout"))
    out, lse = ra.fwd(q, k, v, n, causal, layout)
    dq, dk, dv = ra.bwd(q, k, v, out, lse, do, n, causal, layout)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attn_fwd(x["q"], x["k"], x["v"], n, causal, layout)
    rq, rk, rv = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], n, causal, layout)
    what = f"seed {seed}: B{B} H{H} Hkv{Hkv} L{L} d{d} n{n} {layout} causal={causal} {dtype}"
    assert_close(to_np(out), ref_o, dtype, "out, " + what)
    assert_close(to_np(lse), ref_l, dtype, "lse, " + what)
    for got, ref, name in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        assert_close(to_np(got), ref, dtype, name + ", " + what)
    # one device's block (i, j), written, against the oracle's block
    rng = np.random.default_rng(seed + 1)
    i, j = int(rng.integers(n)), int(rng.integers(n))
    S = L // n
    sh = lambda t, s: t[:, :, s * S:(s + 1) * S].contiguous()
    o_b = torch.full((B, H, S, d), float("nan"), device=DEV)
    l_b = torch.full((B, H, S), float("nan"), device=DEV)
    ra.block_fwd(sh(q, i), sh(k, j), sh(v, j), o_b, l_b, n, i, j, False, causal, layout)
    ro, rl = oracle.block_fwd(sh(x["q"], i), sh(x["k"], j), sh(x["v"], j), L, n, causal, layout, i, j)
    empty = np.isneginf(rl)
    assert np.array_equal(np.isneginf(to_np(l_b)), empty), what
    if (~empty).any():
        assert_close(to_np(o_b)[~empty], ro[~empty], dtype, f"block ({i},{j}) out, " + what)
        assert_close(to_np(l_b)[~empty], rl[~empty], dtype, f"block ({i},{j}) lse, " + what)
