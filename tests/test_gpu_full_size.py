"""Full-size workloads (the sizes the benchmark times), checked on sampled rows the oracle computes
one by one, plus properties that hold at any size."""
import numpy as np
import pytest
import torch

import oracle
import sequence_sharded_exact_gb300 as ra
from sequence_sharded_exact_gb300 import synth
from parity_util import BF16_MAX_ABS, BF16_REL_L2, errors, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _clean_status():
    torch.cuda.set_device(0)
    ra.device_status()
    yield
    assert ra.device_status() == 0, "a bounded wait ran out inside a kernel"


def sampled_rows(w, count, seed):
    """Random rows over all heads, plus the first and last rows of every chunk of the first and
    last head (chunk boundaries, the start of the sequence and the diagonal tiles)."""
    B, H, L, n = w["B"], w["H"], w["L"], w["n"]
    rng = np.random.default_rng(seed)
    rows = set(rng.choice(B * H * L, size=count, replace=False).tolist())
    chunk = L // n // (2 if w["layout"] == "zigzag" else 1)
    for h in (0, H - 1):
        for c in range(L // chunk):
            for r in (c * chunk, c * chunk + 1, c * chunk + chunk - 1):
                rows.add(((B - 1) * H + h) * L + r)
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("name", ["causal_contig_8k", "zigzag_gqa_32k", "zigzag_gqa_128k",
                                  "zigzag_gqa_64k_train", "striped_gqa_128k"])
def test_full_size_forward_sampled_rows(name):
    w = synth.WORKLOADS[name]
    B, H, Hkv, L, d, n = w["B"], w["H"], w["Hkv"], w["L"], w["d"], w["n"]
    x = synth.make_workload(name, device=DEV, gen_device=DEV, with_dout=False)
    assert ra.fwd_path(B, H, Hkv, L, d, n, w["causal"], w["layout"], w["dtype"]) == "tcgen05"
    out, lse = ra.fwd(x["q"], x["k"], x["v"], n, w["causal"], w["layout"])
    torch.cuda.synchronize()
    # properties at any size: finite everywhere, lse bounded by log of the visible count + max score
    assert torch.isfinite(out).all().item() and torch.isfinite(lse).all().item()
    rows = sampled_rows(w, 384, seed=L)
    host = {t: x[t].cpu() for t in ("q", "k", "v")}
    ref_o, ref_l = oracle.attn_fwd_rows(host["q"], host["k"], host["v"], n, w["causal"],
                                        w["layout"], rows)
    got_o = to_np(out.view(-1, d)[torch.from_numpy(rows).to(DEV)])
    got_l = to_np(lse.view(-1)[torch.from_numpy(rows).to(DEV)])
    for got, ref, what in ((got_o, ref_o, "out"), (got_l, ref_l, "lse")):
        ma, rl = errors(got, ref)
        assert ma <= BF16_MAX_ABS and rl <= BF16_REL_L2, f"{name} {what}: {ma:.3e} {rl:.3e}"


def test_full_size_stepwise_matches_fused():
    """At the long-context size the step-by-step ring (ring-step kernel + LSE merge) and the
    fused kernel agree; both are exact attention up to rounding."""
    name = "zigzag_gqa_32k"
    w = synth.WORKLOADS[name]
    x = synth.make_workload(name, device=DEV, gen_device=DEV, with_dout=False)
    o1, l1 = ra.fwd(x["q"], x["k"], x["v"], w["n"], w["causal"], w["layout"])
    o2, l2 = ra.fwd_stepwise(x["q"], x["k"], x["v"], w["n"], w["causal"], w["layout"])
    torch.cuda.synchronize()
    ma, rl = errors(to_np(o2), to_np(o1))
    assert ma <= BF16_MAX_ABS and rl <= BF16_REL_L2
    assert (l1 - l2).abs().max().item() < 1e-3


@pytest.mark.parametrize("name", ["zigzag_gqa_64k_train", "striped_gqa_64k_train"])
def test_full_size_training_backward(name):
    """The training workload (L=65536, n=16, causal, GQA 4:1): dQ on sampled rows and
    dK/dV on the last keys of the sequence (whose visible queries are few enough for the oracle),
    plus identities that hold at any size: sum over keys of dV equals the group's summed dO, and
    the sum over keys of dK vanishes."""
    w = synth.WORKLOADS[name]
    B, H, Hkv, L, d, n = w["B"], w["H"], w["Hkv"], w["L"], w["d"], w["n"]
    x = synth.make_workload(name, device=DEV, gen_device=DEV, with_dout=True)
    assert ra.bwd_path(B, H, Hkv, L, d, n, w["causal"], w["layout"], w["dtype"]) == "tcgen05"
    out, lse = ra.fwd(x["q"], x["k"], x["v"], n, w["causal"], w["layout"])
    dq, dk, dv = ra.bwd(x["q"], x["k"], x["v"], out, lse, x["dout"], n, w["causal"], w["layout"])
    torch.cuda.synchronize()
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all().item()
    G = H // Hkv
    dsum = x["dout"].double().view(B, Hkv, G, L, d).sum(dim=(2, 3))
    assert (dv.double().sum(dim=2) - dsum).abs().max().item() < 0.5
    assert dk.double().sum(dim=2).abs().max().item() < 0.5
    host = {t: x[t].cpu() for t in ("q", "k", "v", "dout")}
    rows = sampled_rows(w, 96, seed=5)
    ref_dq = oracle.attn_bwd_dq_rows(host["q"], host["k"], host["v"], host["dout"], n,
                                     w["causal"], w["layout"], rows)
    got_dq = to_np(dq.view(-1, d)[torch.from_numpy(rows).to(DEV)])
    ma, rl = errors(got_dq, ref_dq)
    assert ma <= BF16_MAX_ABS and rl <= BF16_REL_L2, f"dq {ma:.3e} {rl:.3e}"
    # keys at the last natural positions, in both kv heads at the ends of the head range
    last = [oracle.natural_position(r, L, n, w["layout"]) for r in range(L)]
    order = np.argsort(last)[-24:]
    keys = np.array([((B - 1) * Hkv + g) * L + int(t) for g in (0, Hkv - 1) for t in order])
    ref_dk, ref_dv = oracle.attn_bwd_dkv_rows(host["q"], host["k"], host["v"], host["dout"], n,
                                              w["causal"], w["layout"], keys)
    idx = torch.from_numpy(keys).to(DEV)
    for got, ref, what in ((dk.view(-1, d)[idx], ref_dk, "dk"), (dv.view(-1, d)[idx], ref_dv, "dv")):
        ma, rl = errors(to_np(got), ref)
        assert ma <= BF16_MAX_ABS and rl <= BF16_REL_L2, f"{what} {ma:.3e} {rl:.3e}"


def test_forward_at_262144_tokens_sampled_rows():
    """The largest sequence in the suite: L = 262144 over 16 zigzag shards (positions up to 2^18),
    8 query heads on 2 kv heads; sampled rows (with chunk edges) against the oracle."""
    B, H, Hkv, L, d, n = 1, 8, 2, 262144, 128, 16
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=torch.bfloat16, seed=262144, device=DEV, gen_device=DEV)
    assert ra.fwd_path(B, H, Hkv, L, d, n, True, "zigzag", torch.bfloat16) == "tcgen05"
    out, lse = ra.fwd(x["q"], x["k"], x["v"], n, True, "zigzag")
    torch.cuda.synchronize()
    assert torch.isfinite(out).all().item() and torch.isfinite(lse).all().item()
    w = dict(B=B, H=H, L=L, n=n, layout="zigzag")
    rows = sampled_rows(w, 160, seed=3)
    host = {t: x[t].cpu() for t in ("q", "k", "v")}
    ref_o, ref_l = oracle.attn_fwd_rows(host["q"], host["k"], host["v"], n, True, "zigzag", rows)
    idx = torch.from_numpy(rows).to(DEV)
    for got, ref, what in ((to_np(out.view(-1, d)[idx]), ref_o, "out"), (to_np(lse.view(-1)[idx]), ref_l, "lse")):
        ma, rl = errors(got, ref)
        assert ma <= BF16_MAX_ABS and rl <= BF16_REL_L2, f"{what}: {ma:.3e} {rl:.3e}"
