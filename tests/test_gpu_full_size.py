"""Full-size workloads (the sizes the benchmark times) against the float64 oracle.

Depth of the element-by-element checks, per workload:
  * causal_contig_8k (B2 H8 L8192, contiguous): every element of out and lse;
  * zigzag_gqa_32k (H32 Hkv8 L32768): the first and the last kv-head group in full (4 query heads x
    32768 rows each) plus 4096 seeded rows of the other heads;
  * zigzag_gqa_128k (H32 Hkv8 L131072, 1% of keys x8): one whole query head (131072 rows) plus 4096
    seeded rows over all heads;
  * zigzag_gqa_64k_train (L65536, n16): dQ on 4096 seeded rows; dK and dV on keys of one kv head
    spread over the whole natural range -- natural positions 0-127 (every query of the group sees
    them: the longest accumulations), the first and last key of every chunk, and seeded random keys;
  * the striped workloads, the head-dim-64 workloads and a 262144-token sequence: sampled rows plus
    chunk edges (backward: sampled dQ rows and the last keys' dK/dV).
Every check reports max-abs and relative L2 error per tensor; the bound is the bf16 one (max-abs 2e-2
and relative L2 5e-3, both).  Properties that hold at any size (finite outputs, sum identities of
the gradients) are checked as well."""
import numpy as np
import pytest
import torch

import oracle
import sequence_sharded_exact_gb300 as ra
from sequence_sharded_exact_gb300 import synth
from parity_util import BF16_MAX_ABS, BF16_REL_L2, assert_close, errors, to_np

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _clean_status():
    torch.cuda.set_device(0)
    ra.device_status()
    yield
    assert ra.device_status() == 0, "a bounded wait ran out inside a kernel"


def sampled_rows(w, count, seed, split=False):
    """Random rows over all heads, plus the first and last rows of every chunk of the first and
    last head (chunk boundaries, the start of the sequence and the diagonal tiles).  With split,
    returns (all rows, mask of the uniformly drawn ones)."""
    B, H, L, n = w["B"], w["H"], w["L"], w["n"]
    rng = np.random.default_rng(seed)
    uniform = set(rng.choice(B * H * L, size=count, replace=False).tolist())
    rows = set(uniform)
    chunk = L // n // (2 if w["layout"] == "zigzag" else 1)
    for h in (0, H - 1):
        for c in range(L // chunk):
            for r in (c * chunk, c * chunk + 1, c * chunk + chunk - 1):
                rows.add(((B - 1) * H + h) * L + r)
    rows = np.array(sorted(rows), dtype=np.int64)
    if split:
        return rows, np.array([r in uniform for r in rows])
    return rows


def check_sampled(got, ref, uniform, what):
    """The bf16 bound on sampled rows: max-abs on every checked row, relative L2 (a per-tensor
    statistic) estimated from the uniformly drawn rows only -- the chunk-edge rows include the
    sequence's second and third tokens, whose few visible keys give the largest gradients of the
    tensor, and would dominate a norm over the hand-picked set."""
    ma = float(np.abs(np.asarray(got) - np.asarray(ref)).max())
    _, rl = errors(np.asarray(got)[uniform], np.asarray(ref)[uniform])
    assert ma <= BF16_MAX_ABS and rl <= BF16_REL_L2, f"{what}: max-abs {ma:.3e}, rel-L2 (uniform rows) {rl:.3e}"


def report(capsys, name, what, got, ref):
    """Max-abs and relative L2 error of one tensor, printed to the terminal and checked."""
    ma, rl = errors(got, ref)
    with capsys.disabled():
        print(f"\n[parity] {name} {what}: {np.asarray(ref).size} values, max-abs {ma:.3e}, rel-L2 {rl:.3e}")
    assert ma <= BF16_MAX_ABS and rl <= BF16_REL_L2, f"{name} {what}: max-abs {ma:.3e}, rel-L2 {rl:.3e}"


def head_rows(w, heads):
    """Flat row indices (b*H + h)*L + r of every row of the given query heads (all batches)."""
    B, H, L = w["B"], w["H"], w["L"]
    return np.concatenate([np.arange(((b * H + h) * L), ((b * H + h) * L) + L, dtype=np.int64)
                           for b in range(B) for h in heads])


def test_causal_contig_8k_every_element(capsys):
    name = "causal_contig_8k"
    w = synth.WORKLOADS[name]
    B, H, Hkv, L, d, n = w["B"], w["H"], w["Hkv"], w["L"], w["d"], w["n"]
    x = synth.make_workload(name, device=DEV, gen_device=DEV, with_dout=False)
    assert ra.fwd_path(B, H, Hkv, L, d, n, w["causal"], w["layout"], w["dtype"]) == "tcgen05"
    out, lse = ra.fwd(x["q"], x["k"], x["v"], n, w["causal"], w["layout"])
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.attn_fwd(x["q"].cpu(), x["k"].cpu(), x["v"].cpu(), n, w["causal"], w["layout"])
    report(capsys, name, "out (every element)", to_np(out), ref_o)
    report(capsys, name, "lse (every element)", to_np(lse), ref_l)


def test_zigzag_gqa_32k_full_kv_groups(capsys):
    name = "zigzag_gqa_32k"
    w = synth.WORKLOADS[name]
    B, H, Hkv, L, d, n = w["B"], w["H"], w["Hkv"], w["L"], w["d"], w["n"]
    G = H // Hkv
    x = synth.make_workload(name, device=DEV, gen_device=DEV, with_dout=False)
    out, lse = ra.fwd(x["q"], x["k"], x["v"], n, w["causal"], w["layout"])
    torch.cuda.synchronize()
    host = {t: x[t].cpu() for t in ("q", "k", "v")}
    first, last = list(range(G)), list(range(H - G, H))
    rng = np.random.default_rng(32768)
    others = np.sort(rng.choice(np.arange(G * L, (H - G) * L), size=4096, replace=False))
    for what, rows in (("kv group 0 (heads 0-3, every row)", head_rows(w, first)),
                       (f"kv group {Hkv - 1} (heads {H - G}-{H - 1}, every row)", head_rows(w, last)),
                       ("4096 seeded rows of heads 4-27", others)):
        ref_o, ref_l = oracle.attn_fwd_rows(host["q"], host["k"], host["v"], n, w["causal"], w["layout"], rows)
        idx = torch.from_numpy(rows).to(DEV)
        report(capsys, name, "out, " + what, to_np(out.view(-1, d)[idx]), ref_o)
        report(capsys, name, "lse, " + what, to_np(lse.view(-1)[idx]), ref_l)


def test_zigzag_gqa_128k_full_head_and_rows(capsys):
    name = "zigzag_gqa_128k"
    w = synth.WORKLOADS[name]
    B, H, Hkv, L, d, n = w["B"], w["H"], w["Hkv"], w["L"], w["d"], w["n"]
    x = synth.make_workload(name, device=DEV, gen_device=DEV, with_dout=False)
    out, lse = ra.fwd(x["q"], x["k"], x["v"], n, w["causal"], w["layout"])
    torch.cuda.synchronize()
    assert torch.isfinite(out).all().item() and torch.isfinite(lse).all().item()
    host = {t: x[t].cpu() for t in ("q", "k", "v")}
    rng = np.random.default_rng(131072)
    for what, rows in ((f"head {H - 1} (every row)", head_rows(w, [H - 1])),
                       ("4096 seeded rows of all heads", np.sort(rng.choice(B * H * L, size=4096, replace=False)))):
        ref_o, ref_l = oracle.attn_fwd_rows(host["q"], host["k"], host["v"], n, w["causal"], w["layout"], rows)
        idx = torch.from_numpy(rows).to(DEV)
        report(capsys, name, "out, " + what, to_np(out.view(-1, d)[idx]), ref_o)
        report(capsys, name, "lse, " + what, to_np(lse.view(-1)[idx]), ref_l)


@pytest.mark.parametrize("name", ["zigzag_gqa_64k_train", "striped_gqa_64k_train", "zigzag_gqa_64k_train_d64"])
def test_training_backward_over_the_whole_range(capsys, name):
    """dQ on 4096 seeded rows against the exact gradient; then the most sensitive rows and keys --
    dQ at positions 0-63 of every head, dK and dV on keys of the last kv head at natural positions
    0-127, at the first and last position of every 2048-token chunk (for zigzag, the first keys of
    every shard) and at 64 seeded random positions -- against the backward's definition applied to
    the inputs this backward receives: D = rowsum(dO * out) over the stored bf16 out it is given,
    as the rounded q, k, v are read.  At the first positions a gradient is a sum of a few large,
    cancelling terms, and the rounding of out alone moves it by up to ~1.5e-2 (printed beside)."""
    w = synth.WORKLOADS[name]
    B, H, Hkv, L, d, n = w["B"], w["H"], w["Hkv"], w["L"], w["d"], w["n"]
    x = synth.make_workload(name, device=DEV, gen_device=DEV, with_dout=True)
    assert ra.bwd_path(B, H, Hkv, L, d, n, w["causal"], w["layout"], w["dtype"]) == "tcgen05"
    out, lse = ra.fwd(x["q"], x["k"], x["v"], n, w["causal"], w["layout"])
    dq, dk, dv = ra.bwd(x["q"], x["k"], x["v"], out, lse, x["dout"], n, w["causal"], w["layout"])
    torch.cuda.synchronize()
    host = {t: x[t].cpu() for t in ("q", "k", "v", "dout")}
    out_h = out.cpu()
    rng = np.random.default_rng(65536)
    rows = np.sort(rng.choice(B * H * L, size=4096, replace=False))
    ref_dq = oracle.attn_bwd_dq_rows(host["q"], host["k"], host["v"], host["dout"], n, w["causal"], w["layout"], rows)
    report(capsys, name, "dq, 4096 seeded rows", to_np(dq.view(-1, d)[torch.from_numpy(rows).to(DEV)]), ref_dq)
    # natural position -> buffer row of the layout, from the oracle's own position map
    nat = np.array([oracle.natural_position(r, L, n, w["layout"]) for r in range(L)], dtype=np.int64)
    row_of = np.empty(L, dtype=np.int64)
    row_of[nat] = np.arange(L)
    # the first 64 positions of every head: few visible keys, the largest gradients of the tensor
    # (element-wise bound only: a relative L2 is a per-tensor statistic, estimated above)
    early = np.array([((b * H + h) * L + int(row_of[p])) for b in range(B) for h in range(H) for p in range(64)],
                     dtype=np.int64)
    ref_e = oracle.attn_bwd_dq_rows(host["q"], host["k"], host["v"], host["dout"], n, w["causal"], w["layout"],
                                    early, out=out_h)
    exact_e = oracle.attn_bwd_dq_rows(host["q"], host["k"], host["v"], host["dout"], n, w["causal"],
                                      w["layout"], early)
    got_e = to_np(dq.view(-1, d)[torch.from_numpy(early).to(DEV)])
    ma = float(np.abs(got_e - ref_e).max())
    with capsys.disabled():
        print(f"\n[parity] {name} dq, positions 0-63 of every head: {ref_e.size} values, max-abs {ma:.3e} "
              f"(against the exact gradient: {float(np.abs(got_e - exact_e).max()):.3e})")
    assert ma <= BF16_MAX_ABS, f"dq at early positions: max-abs {ma:.3e}"
    chunk = L // (2 * n)
    positions = set(range(128))
    for c in range(L // chunk):
        positions.update((c * chunk, c * chunk + chunk - 1))
    positions.update(rng.choice(L, size=64, replace=False).tolist())
    g = Hkv - 1
    keys = np.array(sorted(((B - 1) * Hkv + g) * L + int(row_of[p]) for p in positions), dtype=np.int64)
    assert keys.size >= 64
    ref_dk, ref_dv = oracle.attn_bwd_dkv_rows(host["q"], host["k"], host["v"], host["dout"], n, w["causal"],
                                              w["layout"], keys, out=out_h)
    idx = torch.from_numpy(keys).to(DEV)
    what = f"{keys.size} keys of kv head {g} (positions 0-127, every chunk edge, 64 seeded; D from the given out)"
    report(capsys, name, "dk, " + what, to_np(dk.view(-1, d)[idx]), ref_dk)
    report(capsys, name, "dv, " + what, to_np(dv.view(-1, d)[idx]), ref_dv)


@pytest.mark.parametrize("name", ["zigzag_gqa_64k_train", "striped_gqa_128k", "zigzag_gqa_128k_d64"])
def test_full_size_forward_sampled_rows(name):
    w = synth.WORKLOADS[name]
    B, H, Hkv, L, d, n = w["B"], w["H"], w["Hkv"], w["L"], w["d"], w["n"]
    x = synth.make_workload(name, device=DEV, gen_device=DEV, with_dout=False)
    assert ra.fwd_path(B, H, Hkv, L, d, n, w["causal"], w["layout"], w["dtype"]) == "tcgen05"
    out, lse = ra.fwd(x["q"], x["k"], x["v"], n, w["causal"], w["layout"])
    torch.cuda.synchronize()
    # properties at any size: finite everywhere, lse bounded by log of the visible count + max score
    assert torch.isfinite(out).all().item() and torch.isfinite(lse).all().item()
    rows, uniform = sampled_rows(w, 384, seed=L, split=True)
    host = {t: x[t].cpu() for t in ("q", "k", "v")}
    ref_o, ref_l = oracle.attn_fwd_rows(host["q"], host["k"], host["v"], n, w["causal"],
                                        w["layout"], rows)
    got_o = to_np(out.view(-1, d)[torch.from_numpy(rows).to(DEV)])
    got_l = to_np(lse.view(-1)[torch.from_numpy(rows).to(DEV)])
    for got, ref, what in ((got_o, ref_o, "out"), (got_l, ref_l, "lse")):
        check_sampled(got, ref, uniform, f"{name} {what}")


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


@pytest.mark.parametrize("name", ["zigzag_gqa_64k_train", "striped_gqa_64k_train", "zigzag_gqa_64k_train_d64"])
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
    rows, uniform = sampled_rows(w, 96, seed=5, split=True)
    ref_dq = oracle.attn_bwd_dq_rows(host["q"], host["k"], host["v"], host["dout"], n,
                                     w["causal"], w["layout"], rows)
    got_dq = to_np(dq.view(-1, d)[torch.from_numpy(rows).to(DEV)])
    check_sampled(got_dq, ref_dq, uniform, f"{name} dq")
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
    rows, uniform = sampled_rows(w, 160, seed=3, split=True)
    host = {t: x[t].cpu() for t in ("q", "k", "v")}
    ref_o, ref_l = oracle.attn_fwd_rows(host["q"], host["k"], host["v"], n, True, "zigzag", rows)
    idx = torch.from_numpy(rows).to(DEV)
    for got, ref, what in ((to_np(out.view(-1, d)[idx]), ref_o, "out"), (to_np(lse.view(-1)[idx]), ref_l, "lse")):
        check_sampled(got, ref, uniform, what)


def test_million_tokens_forward_dq_and_rope_sampled_rows():
    """A million tokens (L = 2^20) over 32 zigzag shards, 8 query heads on 2 kv heads: the pages'
    long-context case for one device's worth of compute.  Sampled rows of the forward (out, lse) and
    of dQ, with the first, second and last rows of every chunk of the first and last head, against
    the oracle; RoPE of one head in place against the oracle's rotation of every row (positions up
    to 2^20 - 1).  The float32 dQ tensor holds 2^30 elements (4 GiB): byte offsets pass 2^32."""
    B, H, Hkv, L, d, n = 1, 8, 2, 1 << 20, 128, 32
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=torch.bfloat16, seed=1 << 20, with_dout=True,
                          device=DEV, gen_device=DEV)
    assert ra.fwd_path(B, H, Hkv, L, d, n, True, "zigzag", torch.bfloat16) == "tcgen05"
    assert ra.bwd_path(B, H, Hkv, L, d, n, True, "zigzag", torch.bfloat16) == "tcgen05"
    out, lse = ra.fwd(x["q"], x["k"], x["v"], n, True, "zigzag")
    dq, dk, dv = ra.bwd(x["q"], x["k"], x["v"], out, lse, x["dout"], n, True, "zigzag")
    torch.cuda.synchronize()
    for t in (out, lse, dq, dk, dv):
        assert torch.isfinite(t).all().item()
    w = dict(B=B, H=H, L=L, n=n, layout="zigzag")
    rows, uniform = sampled_rows(w, 96, seed=20, split=True)
    host = {t: x[t].cpu() for t in ("q", "k", "v", "dout")}
    ref_o, ref_l = oracle.attn_fwd_rows(host["q"], host["k"], host["v"], n, True, "zigzag", rows)
    ref_dq = oracle.attn_bwd_dq_rows(host["q"], host["k"], host["v"], host["dout"], n, True, "zigzag", rows)
    idx = torch.from_numpy(rows).to(DEV)
    for got, ref, what in ((out.view(-1, d)[idx], ref_o, "out"), (lse.view(-1)[idx], ref_l, "lse"),
                           (dq.view(-1, d)[idx], ref_dq, "dq")):
        check_sampled(to_np(got), ref, uniform, what)
    del out, lse, dq, dk, dv
    # RoPE of the last kv head's keys, every row
    kh = x["k"][:, Hkv - 1:].contiguous()
    ref_r = oracle.rope(kh.cpu(), n, "zigzag")
    ra.rope(kh, n, "zigzag")
    torch.cuda.synchronize()
    assert_close(to_np(kh), ref_r, torch.bfloat16, "rope of 2^20 rows", stored_bf16=True)


def test_float32_output_backward_at_the_first_positions_against_the_exact_gradient(capsys):
    """The striped training workload, where the backward on the stored bf16 output reaches 2.06e-2
    at key position 1 against the exact gradient: with the forward's float32 output kept for D
    (ring_attn_fwd_f32out / ring_attn_bwd_f32out), dQ at positions 0-63 of every head and dK, dV
    on the first 128 keys of the last kv head, against the exact gradient."""
    name = "striped_gqa_64k_train"
    w = synth.WORKLOADS[name]
    B, H, Hkv, L, d, n = w["B"], w["H"], w["Hkv"], w["L"], w["d"], w["n"]
    x = synth.make_workload(name, device=DEV, gen_device=DEV, with_dout=True)
    o32, lse = ra.fwd_f32out(x["q"], x["k"], x["v"], n, w["causal"], w["layout"])
    dq, dk, dv = ra.bwd_f32out(x["q"], x["k"], x["v"], o32, lse, x["dout"], n, w["causal"], w["layout"])
    torch.cuda.synchronize()
    host = {t: x[t].cpu() for t in ("q", "k", "v", "dout")}
    nat = np.array([oracle.natural_position(r, L, n, w["layout"]) for r in range(L)], dtype=np.int64)
    row_of = np.empty(L, dtype=np.int64)
    row_of[nat] = np.arange(L)
    early = np.array([((b * H + h) * L + int(row_of[p])) for b in range(B) for h in range(H) for p in range(64)],
                     dtype=np.int64)
    ref_e = oracle.attn_bwd_dq_rows(host["q"], host["k"], host["v"], host["dout"], n, w["causal"], w["layout"], early)
    got_e = to_np(dq.view(-1, d)[torch.from_numpy(early).to(DEV)])
    ma = float(np.abs(got_e - ref_e).max())
    with capsys.disabled():
        print(f"\n[parity] {name} float32-output backward, dq at positions 0-63: max-abs {ma:.3e} (exact gradient)")
    assert ma <= BF16_MAX_ABS
    g = Hkv - 1
    keys = np.array(sorted(((B - 1) * Hkv + g) * L + int(row_of[p]) for p in range(128)), dtype=np.int64)
    ref_dk, ref_dv = oracle.attn_bwd_dkv_rows(host["q"], host["k"], host["v"], host["dout"], n, w["causal"],
                                              w["layout"], keys)
    idx = torch.from_numpy(keys).to(DEV)
    report(capsys, name, "float32-output backward, dk, keys 0-127 (exact gradient)", to_np(dk.view(-1, d)[idx]), ref_dk)
    report(capsys, name, "float32-output backward, dv, keys 0-127 (exact gradient)", to_np(dv.view(-1, d)[idx]), ref_dv)


def test_training_backward_with_bf16_gradients_at_full_size():
    """The bf16-gradient path at the training size (dQ summed in the float32 workspace, then
    converted; dK, dV rounded in the kernel's epilogue) gives the float32-gradient path's values
    rounded to bf16: dK and dV bit for bit; dQ, whose float32 sums add in arrival order in both runs,
    within one bf16 step plus a floor of 2^-16 of the tensor's largest element for elements whose
    terms cancel (the order of the additions moves their float32 sum by more than their own bf16
    step), and within 2^-8 in relative L2."""
    name = "zigzag_gqa_64k_train"
    w = synth.WORKLOADS[name]
    n = w["n"]
    x = synth.make_workload(name, device=DEV, gen_device=DEV, with_dout=True)
    out, lse = ra.fwd(x["q"], x["k"], x["v"], n, w["causal"], w["layout"])
    f = ra.bwd(x["q"], x["k"], x["v"], out, lse, x["dout"], n, w["causal"], w["layout"])
    h = ra.bwd(x["q"], x["k"], x["v"], out, lse, x["dout"], n, w["causal"], w["layout"], grad_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert all(t.dtype == torch.bfloat16 for t in h)
    assert torch.equal(h[1], f[1].to(torch.bfloat16)) and torch.equal(h[2], f[2].to(torch.bfloat16))
    diff = (h[0].float() - f[0]).abs()
    bound = f[0].abs() * 2.0 ** -7 + f[0].abs().max() * 2.0 ** -16
    assert bool((diff <= bound).all()), f"dq: worst excess {(diff - bound).max().item():.3e}"
    assert (diff.norm() / f[0].norm()).item() <= 2.0 ** -8
