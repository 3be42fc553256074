"""The work the tensor-core kernels do, counted on the device (ring_attn_*_tile_visits): every
(query tile, key tile) pair that holds a visible (query, key) pair is computed exactly once and no
other pair is -- the causal skip of fully masked blocks (M4-051 section 3) -- and the counted runs
give the same results as the plain ones."""
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


def expected_visits(B, H, L, n, causal, layout, q_tile, k_tile=128):
    """Per (query shard, key shard): the (q_tile-row query block, k_tile-row key tile) pairs of
    consecutive buffer rows holding a visible pair, i.e. whose smallest key position does not
    exceed the largest query position (every pair when not causal), times B * H."""
    pos = np.array([oracle.natural_position(r, L, n, layout) for r in range(L)], dtype=np.int64)
    S = L // n
    qmax = pos.reshape(L // q_tile, q_tile).max(axis=1)
    kmin = pos.reshape(L // k_tile, k_tile).min(axis=1)
    vis = kmin[None, :] <= qmax[:, None] if causal else np.ones((qmax.size, kmin.size), bool)
    qs = np.arange(qmax.size) * q_tile // S
    ks = np.arange(kmin.size) * k_tile // S
    out = np.zeros((n, n), np.int64)
    np.add.at(out, (np.repeat(qs, ks.size), np.tile(ks, qs.size)), vis.ravel().astype(np.int64))
    return out * B * H


CASES = [
    # B, H, Hkv, L, n, causal, layout
    (1, 2, 1, 2048, 4, True, "contiguous"),
    (1, 2, 1, 2048, 4, True, "zigzag"),
    (1, 2, 1, 2048, 4, True, "striped"),
    (2, 2, 2, 1024, 2, False, "contiguous"),
    (1, 4, 1, 4096, 8, True, "zigzag"),
]


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("B,H,Hkv,L,n,causal,layout", CASES)
def test_forward_visits_exactly_the_visible_blocks(B, H, Hkv, L, n, causal, layout, d):
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=torch.bfloat16, seed=L + n, device=DEV)
    out, lse, visits = ra.fwd_tile_visits(x["q"], x["k"], x["v"], n, causal, layout)
    out2, lse2 = ra.fwd(x["q"], x["k"], x["v"], n, causal, layout)
    torch.cuda.synchronize()
    exp = expected_visits(B, H, L, n, causal, layout, q_tile=256)
    assert np.array_equal(visits.cpu().numpy(), exp)
    # the forward has no atomics: the counted run is bit-identical to the plain one
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    if causal and layout == "contiguous":
        assert np.all(np.triu(visits.cpu().numpy(), 1) == 0)  # shard i never touches j > i
    if L <= 2048:
        # the same zero pattern as the oracle's ring walk, counted on tokens
        _, _, pairs = oracle.ring_fwd(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), n, causal, layout)
        assert np.array_equal(visits.cpu().numpy() == 0, pairs == 0)


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("B,H,Hkv,L,n,causal,layout", CASES)
def test_backward_visits_exactly_the_visible_tiles(B, H, Hkv, L, n, causal, layout, d):
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=torch.bfloat16, seed=L * 2 + n, with_dout=True,
                          device=DEV)
    q, k, v, do = x["q"], x["k"], x["v"], x["dout"]
    out, lse = ra.fwd(q, k, v, n, causal, layout)
    dq, dk, dv, visits = ra.bwd_tile_visits(q, k, v, out, lse, do, n, causal, layout)
    ref = ra.bwd(q, k, v, out, lse, do, n, causal, layout)
    torch.cuda.synchronize()
    exp = expected_visits(B, H, L, n, causal, layout, q_tile=128)
    assert np.array_equal(visits.cpu().numpy(), exp)
    for g, r, name in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
        assert_close(to_np(g), to_np(r), torch.float32, name, max_abs=1e-4)


def test_long_context_forward_visits():
    """L = 131072, n = 8, zigzag: every shard pair is visited, the counts match the visible
    blocks, and the executed tiles exceed the causal area by under 1 %."""
    w = synth.WORKLOADS["zigzag_gqa_128k"]
    B, H, Hkv, L, n = w["B"], w["H"], w["Hkv"], w["L"], w["n"]
    x = synth.make_workload("zigzag_gqa_128k", device=DEV, gen_device=DEV, with_dout=False)
    _, _, visits = ra.fwd_tile_visits(x["q"], x["k"], x["v"], n, w["causal"], w["layout"])
    torch.cuda.synchronize()
    got = visits.cpu().numpy()
    assert np.array_equal(got, expected_visits(B, H, L, n, True, "zigzag", q_tile=256))
    assert np.all(got > 0)
    causal_area_tiles = B * H * (L * L / 2) / (256 * 128)
    assert 1.0 <= got.sum() / causal_area_tiles < 1.01
