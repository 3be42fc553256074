"""GPU parity of the Ulysses variant: the all-to-all re-layouts bit for bit against a numpy
permutation, and the whole forward against the float64 oracle and the ring forward."""
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


def positions(L, n, layout):
    return np.array([oracle.natural_position(r, L, n, layout) for r in range(L)])


def token_to_head_split(x, n, layout):
    """numpy: [n, B, S, H, d] -> [n, B, H/n, L, d]; local token s of shard i goes to natural
    position p(i*S + s), head h to shard h // (H/n)."""
    n_, B, S, H = x.shape[:4]
    L, Hn = n * S, H // n
    pos = positions(L, n, layout)
    rows = np.moveaxis(x, 0, 1).reshape(B, L, H, *x.shape[4:])  # B, buffer row, H, ...
    out = np.empty((n, B, Hn, L) + x.shape[4:], x.dtype)
    for h in range(H):
        out[h // Hn, :, h % Hn][:, pos] = rows[:, :, h]
    return out


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_a2a_is_the_permutation_both_ways(layout, dtype):
    n, B, S, H, d = 4, 2, 64, 8, 128
    x = torch.arange(n * B * S * H * d, dtype=torch.float32).reshape(n, B, S, H, d).remainder(251).to(dtype)
    hs = ra.ulysses_a2a(x.to(DEV), n, layout, direction=0)
    back = ra.ulysses_a2a(hs, n, layout, direction=1)
    torch.cuda.synchronize()
    ref = token_to_head_split(x.float().numpy(), n, layout)
    assert np.array_equal(hs.float().cpu().numpy(), ref)
    assert torch.equal(back.cpu(), x)


def test_a2a_lse_rows():
    n, B, S, H = 8, 1, 32, 16
    x = torch.randn(n, B, S, H, generator=torch.Generator().manual_seed(1))
    hs = ra.ulysses_a2a(x.to(DEV), n, "zigzag", direction=0)
    torch.cuda.synchronize()
    assert np.array_equal(hs.cpu().numpy(), token_to_head_split(x.numpy(), n, "zigzag"))


def to_token_split(t, n):
    """[B, H, L, d] in the layout's buffer order -> [n, B, S, H, d] (shard i = buffer rows iS..)."""
    B, H, L = t.shape[:3]
    S = L // n
    x = t.reshape(B, H, n, S, *t.shape[3:])
    return np.ascontiguousarray(np.moveaxis(np.moveaxis(x, 2, 0), 2, 3))  # n, B, S, H, ...


CASES = [
    # B, H, Hkv, L, d, n, causal, layout, dtype
    (1, 8, 4, 2048, 128, 4, True, "contiguous", torch.bfloat16),   # tensor-core attention per shard
    (1, 8, 8, 1024, 128, 2, True, "zigzag", torch.bfloat16),
    (2, 4, 4, 1024, 128, 4, False, "striped", torch.bfloat16),
    (1, 4, 2, 512, 64, 2, True, "zigzag", torch.float32),          # CUDA-core attention per shard
]


@pytest.mark.parametrize("B,H,Hkv,L,d,n,causal,layout,dtype", CASES)
def test_ulysses_fwd_matches_oracle(B, H, Hkv, L, d, n, causal, layout, dtype):
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=dtype, seed=L + H)
    q, k, v = (torch.from_numpy(to_token_split(x[t].float().numpy(), n)).to(dtype) for t in ("q", "k", "v"))
    out, lse = ra.ulysses_fwd(q.to(DEV), k.to(DEV), v.to(DEV), n, causal, layout)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attn_fwd(x["q"], x["k"], x["v"], n, causal, layout)
    assert_close(to_np(out), to_token_split(ref_o, n), dtype, "out")
    assert_close(to_np(lse), to_token_split(ref_l, n), dtype, "lse")


def test_ulysses_equals_ring_on_the_long_context_workload():
    """L = 131072, 32 query / 8 kv heads over 8 shards: the Ulysses forward (4 query heads and one
    kv head per shard) and the zigzag ring forward agree on every row."""
    w = synth.WORKLOADS["zigzag_gqa_128k"]
    B, H, Hkv, L, d, n = w["B"], w["H"], w["Hkv"], w["L"], w["d"], w["n"]
    x = synth.make_workload("zigzag_gqa_128k", device=DEV, gen_device=DEV, with_dout=False)
    o_ring, l_ring = ra.fwd(x["q"], x["k"], x["v"], n, True, "zigzag")
    tok = lambda t: t.view(B, t.shape[1], n, L // n, d).permute(2, 0, 3, 1, 4).contiguous()
    o_u, l_u = ra.ulysses_fwd(tok(x["q"]), tok(x["k"]), tok(x["v"]), n, True, "zigzag")
    torch.cuda.synchronize()
    o_ring_tok = tok(o_ring)
    l_ring_tok = l_ring.view(B, H, n, L // n).permute(2, 0, 3, 1)
    # each output is within 2e-2 + 2^-9 |x| (bf16 storage) of exact attention, so they differ by at
    # most twice that
    excess = ((o_u.float() - o_ring_tok.float()).abs() - (4e-2 + o_ring_tok.float().abs() * 2.0 ** -8)).max().item()
    assert excess <= 0, excess
    assert (l_u - l_ring_tok).abs().max().item() < 1e-3
    # and sampled rows of the Ulysses output against the oracle, one by one
    rng = np.random.default_rng(7)
    rows = np.sort(rng.choice(B * H * L, size=256, replace=False))
    host = {t: x[t].cpu() for t in ("q", "k", "v")}
    ref_o, ref_l = oracle.attn_fwd_rows(host["q"], host["k"], host["v"], n, True, "zigzag", rows)
    o_buf = o_u.permute(1, 3, 0, 2, 4).reshape(B * H * L, d)  # back to [B][H][L] buffer order
    l_buf = l_u.permute(1, 3, 0, 2).reshape(-1)
    idx = torch.from_numpy(rows).to(DEV)
    assert_close(to_np(o_buf[idx]), ref_o, torch.bfloat16, "sampled out")
    assert_close(to_np(l_buf[idx]), ref_l, torch.bfloat16, "sampled lse")


@pytest.mark.parametrize("B,H,Hkv,L,d,n,causal,layout,dtype", [
    (1, 8, 4, 1024, 128, 4, True, "zigzag", torch.bfloat16),    # tensor-core backward per shard
    (1, 4, 4, 512, 128, 2, False, "contiguous", torch.bfloat16),
    (1, 4, 2, 384, 64, 2, True, "striped", torch.float32),      # CUDA-core backward per shard
])
@pytest.mark.parametrize("grad_dtype", [torch.float32, torch.bfloat16])
def test_ulysses_bwd_matches_oracle(B, H, Hkv, L, d, n, causal, layout, dtype, grad_dtype):
    if dtype == torch.float32 and grad_dtype == torch.bfloat16:
        pytest.skip("bf16 gradients are only offered for bf16 inputs in this suite")
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=dtype, seed=L + 7 * H, with_dout=True)
    tok = {t: torch.from_numpy(to_token_split(x[t].float().numpy(), n)).to(dtype).to(DEV)
           for t in ("q", "k", "v", "dout")}
    out, lse = ra.ulysses_fwd(tok["q"], tok["k"], tok["v"], n, causal, layout)
    dq, dk, dv = ra.ulysses_bwd(tok["q"], tok["k"], tok["v"], out, lse, tok["dout"], n, causal, layout,
                                grad_dtype=grad_dtype)
    torch.cuda.synchronize()
    rq, rk, rv = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], n, causal, layout)
    for got, ref, name in ((dq, rq, "dq"), (dk, rk, "dk"), (dv, rv, "dv")):
        assert got.dtype == grad_dtype
        assert_close(to_np(got), to_token_split(ref, n), dtype, name, stored_bf16=grad_dtype == torch.bfloat16)
