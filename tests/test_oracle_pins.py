"""Pins of the float64 oracle against what the pages and the mathematics fix (CPU only).

Each test checks the oracle against something other than itself: a library routine on a special
case that reduces to it (torch float64 scaled_dot_product_attention and autograd), closed forms,
invariants the Ring Attention pages state (n-step ring result equals full attention; causal shard i
needs only blocks j <= i; zigzag equalises per-shard work, contiguous work grows with i; constant V
gives a constant output), special cases with known answers, and central finite differences.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from sequence_sharded_exact_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def buffer_to_natural(L, n, layout):
    """Natural position of every buffer row, built as a concatenation of shard-local ranges.

    Contiguous: shard i is natural range [i*S, (i+1)*S).  Zigzag: 2n chunks of C tokens; shard i is
    chunk i followed by chunk 2n-1-i (airsota M4-051, section 4 item 2)."""
    if layout == "contiguous":
        return np.arange(L)
    if layout == "striped":  # shard i: tokens i, i + n, i + 2n, ... (Lecture 30, section 3.2)
        return np.concatenate([np.arange(i, L, n) for i in range(n)])
    C = L // (2 * n)
    parts = []
    for i in range(n):
        parts.append(np.arange(i * C, (i + 1) * C))
        mirror = 2 * n - 1 - i
        parts.append(np.arange(mirror * C, (mirror + 1) * C))
    return np.concatenate(parts)


def to_natural(x, perm):
    """Rows of a [.., L, ..] buffer (sequence axis 2) rearranged into natural order."""
    out = np.empty_like(x)
    out[:, :, perm] = x
    return out


def sdpa64(q, k, v, causal):
    """torch float64 library attention on natural-order inputs: (out, lse)."""
    qt, kt, vt = (torch.from_numpy(np.asarray(a, np.float64)) for a in (q, k, v))
    G = qt.shape[1] // kt.shape[1]
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=causal,
                                                           enable_gqa=G > 1)
    kr = kt.repeat_interleave(G, dim=1)
    s = torch.matmul(qt, kr.transpose(-1, -2)) / math.sqrt(qt.shape[-1])
    if causal:
        L = qt.shape[2]
        s = s.masked_fill(torch.ones(L, L, dtype=torch.bool).triu(1), float("-inf"))
    return out.numpy(), torch.logsumexp(s, dim=-1).numpy()


def rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape).astype(np.float32)


SMALL_CASES = [
    # (B, H, Hkv, L, d, n, causal, layout)
    (1, 1, 1, 16, 8, 1, False, "contiguous"),
    (1, 2, 1, 16, 8, 2, True, "contiguous"),
    (2, 4, 2, 24, 4, 3, True, "zigzag"),
    (1, 4, 1, 32, 8, 4, True, "zigzag"),
    (1, 2, 2, 32, 8, 8, False, "zigzag"),
    (2, 3, 3, 30, 5, 5, True, "contiguous"),
    (1, 4, 4, 32, 8, 16, True, "zigzag"),
    (1, 2, 1, 24, 8, 4, True, "striped"),
    (2, 4, 2, 30, 4, 5, True, "striped"),
    (1, 2, 2, 32, 8, 8, False, "striped"),
]


@pytest.mark.parametrize("B,H,Hkv,L,d,n,causal,layout", SMALL_CASES)
def test_fwd_matches_library_attention(B, H, Hkv, L, d, n, causal, layout):
    """Brute-force pin: the oracle equals torch float64 SDPA after undoing the layout."""
    q, k, v = rand((B, H, L, d), 1), rand((B, Hkv, L, d), 2), rand((B, Hkv, L, d), 3)
    out, lse = oracle.attn_fwd(q, k, v, n, causal, layout)
    perm = buffer_to_natural(L, n, layout)
    ref_out, ref_lse = sdpa64(to_natural(q, perm), to_natural(k, perm), to_natural(v, perm), causal)
    np.testing.assert_allclose(to_natural(out, perm), ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(to_natural(lse[..., None], perm)[..., 0], ref_lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("L,n,layout", [(16, 1, "contiguous"), (24, 3, "zigzag"), (64, 8, "zigzag"),
                                        (40, 5, "contiguous"), (32, 16, "zigzag"), (24, 4, "striped"),
                                        (30, 5, "striped"), (16, 1, "striped")])
def test_natural_position_is_a_permutation(L, n, layout):
    got = np.array([oracle.natural_position(r, L, n, layout) for r in range(L)])
    np.testing.assert_array_equal(got, buffer_to_natural(L, n, layout))


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
@pytest.mark.parametrize("causal", [False, True])
def test_ring_result_independent_of_n(layout, causal):
    """The n-step ring equals full attention and does not depend on n (M4-051 section 3)."""
    B, H, Hkv, L, d = 1, 4, 2, 64, 8
    qn, kn, vn = rand((B, H, L, d), 11), rand((B, Hkv, L, d), 12), rand((B, Hkv, L, d), 13)
    ref_out, ref_lse = sdpa64(qn, kn, vn, causal)
    for n in (1, 2, 4, 8, 16):
        if layout == "zigzag" and L % (2 * n):
            continue
        perm = buffer_to_natural(L, n, layout)
        q, k, v = qn[:, :, perm], kn[:, :, perm], vn[:, :, perm]
        out, lse, _ = oracle.ring_fwd(q, k, v, n, causal, layout)
        np.testing.assert_allclose(to_natural(out, perm), ref_out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(to_natural(lse[..., None], perm)[..., 0], ref_lse, rtol=0,
                                   atol=1e-12)
        full_out, full_lse = oracle.attn_fwd(q, k, v, n, causal, layout)
        np.testing.assert_allclose(out, full_out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, full_lse, rtol=0, atol=1e-12)


def test_causal_contiguous_uses_only_earlier_blocks():
    """Causal, contiguous: shard i touches blocks j <= i only; pair counts follow S^2 / S(S+1)/2."""
    B, H, Hkv, L, d, n = 1, 2, 1, 48, 4, 6
    S = L // n
    q, k, v = rand((B, H, L, d), 21), rand((B, Hkv, L, d), 22), rand((B, Hkv, L, d), 23)
    _, _, pairs = oracle.ring_fwd(q, k, v, n, True, "contiguous")
    for i in range(n):
        for j in range(n):
            expect = 0 if j > i else (S * S if j < i else S * (S + 1) // 2)
            assert pairs[i, j] == expect * B * H, (i, j)


def test_causal_striped_pair_counts():
    """Striped: block (i, j) holds S(S+1)/2 visible pairs when j <= i and S(S-1)/2 when j > i, so
    every ring step does the same work on every shard."""
    B, H, Hkv, L, d, n = 1, 1, 1, 40, 4, 5
    S = L // n
    q, k, v = rand((B, H, L, d), 34), rand((B, Hkv, L, d), 35), rand((B, Hkv, L, d), 36)
    _, _, pairs = oracle.ring_fwd(q, k, v, n, True, "striped")
    for i in range(n):
        for j in range(n):
            assert pairs[i, j] == (S * (S + 1) // 2 if j <= i else S * (S - 1) // 2), (i, j)


def test_causal_zigzag_pair_counts_are_balanced():
    """Zigzag: every off-diagonal step does half a shard pair (2C^2); every shard the same total."""
    B, H, Hkv, L, d, n = 1, 1, 1, 64, 4, 4
    C = L // (2 * n)
    q, k, v = rand((B, H, L, d), 31), rand((B, Hkv, L, d), 32), rand((B, Hkv, L, d), 33)
    _, _, pairs = oracle.ring_fwd(q, k, v, n, True, "zigzag")
    for i in range(n):
        for j in range(n):
            expect = 2 * C * C if i != j else C * C + C * (C + 1)
            assert pairs[i, j] == expect, (i, j)
    totals = pairs.sum(axis=1)
    assert (totals == totals[0]).all()
    assert totals[0] == (2 * n - 1) * C * C + C * (C + 1)


@pytest.mark.parametrize("L,n,T", [(8192, 8, 128), (2048, 4, 128), (1024, 8, 64), (4096, 2, 256)])
def test_tile_counts_closed_forms(L, n, T):
    """Contiguous shard i: s^2 i + s(s+1)/2; zigzag: (2n-1)c^2 + c(c+1) for every shard."""
    s = L // n // T
    got = oracle.shard_tiles(L, n, True, "contiguous", T)
    np.testing.assert_array_equal(got, [s * s * i + s * (s + 1) // 2 for i in range(n)])
    c = L // (2 * n) // T
    got = oracle.shard_tiles(L, n, True, "zigzag", T)
    np.testing.assert_array_equal(got, [(2 * n - 1) * c * c + c * (c + 1)] * n)
    np.testing.assert_array_equal(oracle.shard_tiles(L, n, False, "zigzag", T), [s * n * s] * n)
    # striped: query tile a of shard i sees key tile b of every shard iff b <= a
    np.testing.assert_array_equal(oracle.shard_tiles(L, n, True, "striped", T), [n * s * (s + 1) // 2] * n)


def test_tile_counts_golden():
    """Sizes the pages state (128K tokens over 8 devices, 16K each, block 128) and the counts the
    oracle's brute-force tile counter produced for the benchmark workloads (written by
    tests/golden/make_golden.py, which calls only the oracle)."""
    with open(os.path.join(GOLDEN, "shard_tiles.json")) as f:
        gold = json.load(f)
    for case in gold["cases"]:
        got = oracle.shard_tiles(case["L"], case["n"], case["causal"], case["layout"], case["tile"])
        assert got.tolist() == case["tiles_per_shard"], case["name"]
    page = gold["page_sizes"]
    assert page["L"] // page["n"] == page["tokens_per_device"]


def test_contiguous_causal_imbalance_ratio():
    """Naive contiguous causal split: last shard's work over first shard's (tile level)."""
    got = oracle.shard_tiles(8192, 8, True, "contiguous", 128)
    assert got[0] == 36 and got[-1] == 484
    assert abs(got.max() / got.mean() - 484 / 260) < 1e-12


def test_constant_v_gives_constant_output():
    B, H, Hkv, L, d, n = 1, 4, 2, 32, 8, 4
    q, k = rand((B, H, L, d), 41), rand((B, Hkv, L, d), 42)
    c = rand((d,), 43)
    v = np.broadcast_to(c, (B, Hkv, L, d)).copy()
    for causal in (False, True):
        for layout in ("contiguous", "zigzag"):
            out, _ = oracle.attn_fwd(q, k, v, n, causal, layout)
            np.testing.assert_allclose(out, np.broadcast_to(c, out.shape), rtol=0, atol=1e-12)
            dout = rand((B, H, L, d), 44)
            dq, dk, dv = oracle.attn_bwd(q, k, v, dout, n, causal, layout)
            np.testing.assert_allclose(dq, 0, atol=1e-12)
            np.testing.assert_allclose(dk, 0, atol=1e-12)


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
def test_closed_form_special_cases(layout):
    B, H, Hkv, L, d, n = 1, 2, 1, 32, 8, 4
    q, k, v = rand((B, H, L, d), 51), rand((B, Hkv, L, d), 52), rand((B, Hkv, L, d), 53)
    perm = buffer_to_natural(L, n, layout)
    r0 = int(np.nonzero(perm == 0)[0][0])  # buffer row of natural position 0
    out, lse = oracle.attn_fwd(q, k, v, n, True, layout)
    # causal row at position 0 sees only itself
    for h in range(H):
        np.testing.assert_allclose(out[0, h, r0], v[0, 0, r0], rtol=0, atol=1e-12)
        s00 = float(np.dot(q[0, h, r0].astype(np.float64), k[0, 0, r0].astype(np.float64))) / math.sqrt(d)
        assert abs(lse[0, h, r0] - s00) < 1e-12
    # Q = 0: uniform weights over the visible keys
    qz = np.zeros_like(q)
    out, lse = oracle.attn_fwd(qz, k, v, n, True, layout)
    vn = v[0, 0][np.argsort(perm)]  # natural-order values
    for r in range(L):
        p = perm[r]
        np.testing.assert_allclose(out[0, 1, r], vn[: p + 1].astype(np.float64).mean(axis=0),
                                   rtol=0, atol=1e-12)
        assert abs(lse[0, 1, r] - math.log(p + 1)) < 1e-12
    out, lse = oracle.attn_fwd(qz, k, v, n, False, layout)
    np.testing.assert_allclose(lse, math.log(L), rtol=0, atol=1e-12)


def test_fwd_rows_match_full():
    B, H, Hkv, L, d, n = 2, 4, 2, 48, 8, 3
    q, k, v = rand((B, H, L, d), 61), rand((B, Hkv, L, d), 62), rand((B, Hkv, L, d), 63)
    out, lse = oracle.attn_fwd(q, k, v, n, True, "zigzag")
    rows = np.array([0, 5, 47, 48 * 3 + 7, B * H * L - 1])
    o2, l2 = oracle.attn_fwd_rows(q, k, v, n, True, "zigzag", rows)
    np.testing.assert_array_equal(o2, out.reshape(-1, d)[rows])
    np.testing.assert_array_equal(l2, lse.reshape(-1)[rows])


@pytest.mark.parametrize("B,H,Hkv,L,d,n,causal,layout", SMALL_CASES)
def test_bwd_matches_library_autograd(B, H, Hkv, L, d, n, causal, layout):
    """Backward pin: torch float64 autograd through SDPA, after undoing the layout."""
    q, k, v, do = (rand(s, i) for i, s in enumerate(
        [(B, H, L, d), (B, Hkv, L, d), (B, Hkv, L, d), (B, H, L, d)], start=71))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, n, causal, layout)
    perm = buffer_to_natural(L, n, layout)
    tq, tk, tv = (torch.from_numpy(to_natural(a, perm).astype(np.float64)).requires_grad_()
                  for a in (q, k, v))
    G = H // Hkv
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                           enable_gqa=G > 1)
    out.backward(torch.from_numpy(to_natural(do, perm).astype(np.float64)))
    np.testing.assert_allclose(to_natural(dq, perm), tq.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(to_natural(dk, perm), tk.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(to_natural(dv, perm), tv.grad.numpy(), rtol=0, atol=1e-11)


def test_bwd_finite_differences():
    """Central differences of sum(out * dout) in float64 on a tiny problem."""
    B, H, Hkv, L, d, n = 1, 2, 1, 8, 4, 2
    q, k, v, do = (rand(s, i).astype(np.float64) for i, s in enumerate(
        [(B, H, L, d), (B, Hkv, L, d), (B, Hkv, L, d), (B, H, L, d)], start=81))
    causal, layout = True, "zigzag"
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, n, causal, layout)
    # The oracle reads float32 inputs, so perturb by a float32-exact step and use its own forward.
    h = 2.0 ** -10

    def f(qq, kk, vv):
        out, _ = oracle.attn_fwd(qq, kk, vv, n, causal, layout)
        return float((out * do).sum())

    q, k, v = (a.astype(np.float32) for a in (q, k, v))
    for name, arr, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for idx in [(0, 0, 0, 0), (0, 0, 3, 1), (0, arr.shape[1] - 1, L - 1, d - 1), (0, 0, 5, 2)]:
            plus, minus = arr.copy(), arr.copy()
            plus[idx] += h
            minus[idx] -= h
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = plus, minus
            num = (f(**{"qq": args_p["q"], "kk": args_p["k"], "vv": args_p["v"]}) -
                   f(**{"qq": args_m["q"], "kk": args_m["k"], "vv": args_m["v"]})) / (2 * h)
            assert abs(num - grad[idx]) <= 1e-5 * max(1.0, abs(grad[idx])), (name, idx, num,
                                                                              grad[idx])


def test_bwd_sum_identities_and_layout_independence():
    B, H, Hkv, L, d = 1, 4, 2, 32, 8
    qn, kn, vn, don = (rand(s, i) for i, s in enumerate(
        [(B, H, L, d), (B, Hkv, L, d), (B, Hkv, L, d), (B, H, L, d)], start=91))
    ref = None
    for n, layout in ((1, "contiguous"), (4, "contiguous"), (2, "zigzag"), (4, "zigzag"),
                      (8, "zigzag"), (4, "striped"), (8, "striped")):
        perm = buffer_to_natural(L, n, layout)
        q, k, v, do = (a[:, :, perm] for a in (qn, kn, vn, don))
        dq, dk, dv = oracle.attn_bwd(q, k, v, do, n, True, layout)
        # sum_t dV_t = sum over the group's query heads of sum_p dO_p (softmax rows sum to one)
        G = H // Hkv
        for g in range(Hkv):
            np.testing.assert_allclose(dv[0, g].sum(axis=0),
                                       do[0, g * G:(g + 1) * G].astype(np.float64).sum(axis=(0, 1)),
                                       atol=1e-11)
            np.testing.assert_allclose(dk[0, g].sum(axis=0), 0, atol=1e-11)
        nat = tuple(to_natural(x, perm) for x in (dq, dk, dv))
        if ref is None:
            ref = nat
        else:
            for a, b in zip(nat, ref):
                np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)


def test_bwd_rows_match_full():
    B, H, Hkv, L, d, n = 1, 4, 2, 32, 8, 4
    q, k, v, do = (rand(s, i) for i, s in enumerate(
        [(B, H, L, d), (B, Hkv, L, d), (B, Hkv, L, d), (B, H, L, d)], start=101))
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, n, True, "zigzag")
    rows = np.array([0, 7, 31, 32 * 2 + 5, B * H * L - 1])
    np.testing.assert_allclose(oracle.attn_bwd_dq_rows(q, k, v, do, n, True, "zigzag", rows),
                               dq.reshape(-1, d)[rows], rtol=0, atol=1e-13)
    keys = np.array([0, 9, 31, 32 + 3, B * Hkv * L - 1])
    dk2, dv2 = oracle.attn_bwd_dkv_rows(q, k, v, do, n, True, "zigzag", keys)
    np.testing.assert_allclose(dk2, dk.reshape(-1, d)[keys], rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv2, dv.reshape(-1, d)[keys], rtol=0, atol=1e-13)


def test_bwd_rows_with_the_exact_output_given_equal_the_definition():
    """D from a given output: given the forward definition's own output (rounded to float32, the
    oracle's input precision), the rows equal the default ones up to that rounding."""
    B, H, Hkv, L, d, n = 1, 4, 2, 32, 8, 4
    q, k, v, do = (rand(s, i) for i, s in enumerate(
        [(B, H, L, d), (B, Hkv, L, d), (B, Hkv, L, d), (B, H, L, d)], start=131))
    o, _ = oracle.attn_fwd(q, k, v, n, True, "zigzag")
    rows = np.arange(B * H * L)
    keys = np.arange(B * Hkv * L)
    np.testing.assert_allclose(oracle.attn_bwd_dq_rows(q, k, v, do, n, True, "zigzag", rows, out=o),
                               oracle.attn_bwd_dq_rows(q, k, v, do, n, True, "zigzag", rows), rtol=0, atol=1e-6)
    dk1, dv1 = oracle.attn_bwd_dkv_rows(q, k, v, do, n, True, "zigzag", keys, out=o)
    dk0, dv0 = oracle.attn_bwd_dkv_rows(q, k, v, do, n, True, "zigzag", keys)
    np.testing.assert_allclose(dk1, dk0, rtol=0, atol=1e-6)
    assert np.array_equal(dv1, dv0)  # dV does not involve D


@pytest.mark.parametrize("layout", ["zigzag", "striped"])
def test_bwd_rows_given_output_enters_only_through_D(layout):
    """Changing one element out[p, c] by delta changes D_p by delta * dO[p, c], and nothing else:
    dV stays the same, dK_t moves by -scale P_pt D-change q_p for every key t that query p sees,
    dQ_p by -scale D-change sum_t P_pt k_t, and every other dQ row stays the same.  P is computed
    here from q, k and the oracle's lse with numpy."""
    B, H, Hkv, L, d, n = 1, 2, 1, 32, 8, 2
    q, k, v, do = (rand(s, i) for i, s in enumerate(
        [(B, H, L, d), (B, Hkv, L, d), (B, Hkv, L, d), (B, H, L, d)], start=141))
    o, lse = oracle.attn_fwd(q, k, v, n, True, layout)
    o = o.astype(np.float32)
    h, r, c, delta = 1, 21, 3, 0.25
    o2 = o.copy()
    o2[0, h, r, c] += delta
    rows = np.arange(B * H * L)
    keys = np.arange(B * Hkv * L)
    dq1 = oracle.attn_bwd_dq_rows(q, k, v, do, n, True, layout, rows, out=o)
    dq2 = oracle.attn_bwd_dq_rows(q, k, v, do, n, True, layout, rows, out=o2)
    dk1, dv1 = oracle.attn_bwd_dkv_rows(q, k, v, do, n, True, layout, keys, out=o)
    dk2, dv2 = oracle.attn_bwd_dkv_rows(q, k, v, do, n, True, layout, keys, out=o2)
    scale = 1.0 / math.sqrt(d)
    nat = buffer_to_natural(L, n, layout)
    qd, kd = q.astype(np.float64), k.astype(np.float64)
    P = np.exp(scale * kd[0, 0] @ qd[0, h, r] - lse[0, h, r]) * (nat <= nat[r])  # [L] over key rows
    dD = delta * float(do[0, h, r, c])
    assert np.array_equal(dv2, dv1)
    np.testing.assert_allclose(dk2 - dk1, -scale * dD * P[:, None] * qd[0, h, r][None, :], rtol=0, atol=1e-12)
    flat = h * L + r
    np.testing.assert_allclose(dq2[flat] - dq1[flat], -scale * dD * (P @ kd[0, 0]), rtol=0, atol=1e-12)
    others = np.arange(B * H * L) != flat
    assert np.array_equal(dq2[others], dq1[others])


def test_synth_recipe():
    """The generator is seeded, rounds to the dtype, and scales exactly round(0.01 L) key rows."""
    a = synth.make_inputs(1, 2, 1, 1000, 8, dtype=torch.bfloat16, seed=7, spike_frac=0.01)
    b = synth.make_inputs(1, 2, 1, 1000, 8, dtype=torch.bfloat16, seed=7, spike_frac=0.01)
    assert all(torch.equal(a[x], b[x]) for x in a)
    plain = synth.make_inputs(1, 2, 1, 1000, 8, dtype=torch.float32, seed=7, spike_frac=0.0)
    spiked = synth.make_inputs(1, 2, 1, 1000, 8, dtype=torch.float32, seed=7, spike_frac=0.01)
    changed = (plain["k"] != spiked["k"]).any(dim=-1).sum().item()
    assert changed == 10
    assert a["q"].dtype == torch.bfloat16


# ------------------------------------------------------------------------------------------------
# Rotary positions (reading C17: natural positions follow the rows; C18: RoFormer pair rotation)
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("layout,n", [("contiguous", 4), ("zigzag", 4), ("striped", 4), ("zigzag", 1)])
def test_rope_is_complex_multiplication_by_natural_position(layout, n):
    """Pair (x0, x1) as the complex number x0 + i x1 is multiplied by exp(i p theta_j),
    theta_j = base^(-2j/d), p = the row's natural position (numpy complex128 exponential)."""
    L, d, base = 32, 8, 500.0
    x = rand((2, 3, L, d), 201)
    y = oracle.rope(x, n, layout, base=base)
    pos = buffer_to_natural(L, n, layout)
    theta = base ** (-np.arange(d // 2) * 2.0 / d)
    z = x[..., 0::2].astype(np.float64) + 1j * x[..., 1::2].astype(np.float64)
    rot = z * np.exp(1j * pos[:, None] * theta[None, :])
    np.testing.assert_allclose(y[..., 0::2], rot.real, rtol=0, atol=1e-12)
    np.testing.assert_allclose(y[..., 1::2], rot.imag, rtol=0, atol=1e-12)


def test_rope_identity_at_position_zero_and_norms():
    L, d = 16, 16
    x = rand((1, 2, L, d), 202)
    y = oracle.rope(x, 2, "contiguous")
    np.testing.assert_array_equal(y[:, :, 0], x[:, :, 0].astype(np.float64))  # p = 0: angle 0
    pair = lambda a: a[..., 0::2] ** 2 + a[..., 1::2] ** 2
    np.testing.assert_allclose(pair(y), pair(x.astype(np.float64)), rtol=1e-12, atol=1e-12)


def test_rope_inverse_undoes_forward():
    L, d = 24, 8
    x = rand((1, 1, L, d), 203).astype(np.float64)
    for layout, n in (("contiguous", 3), ("zigzag", 3), ("striped", 3)):
        fwd = oracle.rope(x, n, layout)
        # forward rotation of x (exact float32 input) then the inverse in float64 by the transpose
        inv_of_x = oracle.rope(x, n, layout, inverse=True)
        # <R x, R x'> = <x, x'> and R^T R = I: check via the bilinear identity on random pairs
        xp = rand((1, 1, L, d), 204)
        lhs = (fwd * oracle.rope(xp, n, layout)).sum(axis=-1)
        np.testing.assert_allclose(lhs, (x * xp).sum(axis=-1), rtol=1e-12, atol=1e-12)
        rhs = (inv_of_x * xp).sum(axis=-1)
        np.testing.assert_allclose(rhs, (x * oracle.rope(xp, n, layout)).sum(axis=-1), rtol=1e-12, atol=1e-12)


def test_rope_scores_depend_on_relative_position_only():
    """<R(p) q, R(t) k> is unchanged when both positions move by the same shift s (the property
    that lets K/V blocks travel with their positions)."""
    L, d = 64, 16
    q1, k1 = rand((d,), 205), rand((d,), 206)
    base_pairs = [(5, 2), (9, 9), (20, 3)]
    for shift in (1, 17, 40):
        for p, t in base_pairs:
            xq = np.zeros((1, 1, L, d), np.float32)
            xk = np.zeros((1, 1, L, d), np.float32)
            xq[0, 0, p], xk[0, 0, t] = q1, k1
            s0 = float((oracle.rope(xq, 1, "contiguous")[0, 0, p] * oracle.rope(xk, 1, "contiguous")[0, 0, t]).sum())
            xq2, xk2 = np.zeros_like(xq), np.zeros_like(xk)
            xq2[0, 0, p + shift], xk2[0, 0, t + shift] = q1, k1
            s1 = float((oracle.rope(xq2, 1, "contiguous")[0, 0, p + shift] *
                        oracle.rope(xk2, 1, "contiguous")[0, 0, t + shift]).sum())
            assert abs(s0 - s1) <= 1e-11 * max(1.0, abs(s0)), (shift, p, t, s0, s1)


def test_rope_layout_equivariance():
    """Rotating a sharded buffer equals rotating the natural-order sequence, then sharding."""
    L, d = 32, 8
    xn = rand((2, 2, L, d), 207)
    yn = oracle.rope(xn, 1, "contiguous")
    for layout, n in (("zigzag", 4), ("striped", 4), ("contiguous", 4)):
        perm = buffer_to_natural(L, n, layout)
        np.testing.assert_array_equal(oracle.rope(xn[:, :, perm], n, layout), yn[:, :, perm])


def test_rope_attention_gradient_chain_matches_autograd():
    """d/dq of sum(attn(R q, R k, v) * dout) = R^T (attention's dQ at the rotated inputs), and the
    same for k: the oracle's chain (attention backward at the rotated inputs, then the inverse
    rotation) against torch float64 autograd through a rotation written as a complex product and
    scaled_dot_product_attention, in natural order."""
    B, H, Hkv, L, d, n = 1, 4, 2, 32, 8, 4
    causal, layout, base = True, "zigzag", 100.0
    q, k, v, do = (rand(s, i) for i, s in enumerate(
        [(B, H, L, d), (B, Hkv, L, d), (B, Hkv, L, d), (B, H, L, d)], start=211))
    qr = oracle.rope(q, n, layout, base=base).astype(np.float32)
    kr = oracle.rope(k, n, layout, base=base).astype(np.float32)
    dq_r, dk_r, _ = oracle.attn_bwd(qr, kr, v, do, n, causal, layout)
    dq = oracle.rope(dq_r, n, layout, base=base, inverse=True)
    dk = oracle.rope(dk_r, n, layout, base=base, inverse=True)

    perm = buffer_to_natural(L, n, layout)
    inv = np.argsort(perm)
    nat = lambda a: torch.from_numpy(a[:, :, inv].astype(np.float64))
    tq, tk, tv, tdo = nat(q).requires_grad_(True), nat(k).requires_grad_(True), nat(v), nat(do)
    theta = torch.tensor(base ** (-np.arange(d // 2) * 2.0 / d), dtype=torch.float64)
    rot = torch.polar(torch.ones(L, d // 2, dtype=torch.float64), torch.arange(L, dtype=torch.float64)[:, None] * theta)

    def rotate(x):
        xc = torch.view_as_complex(x.reshape(*x.shape[:-1], d // 2, 2).contiguous())
        return torch.view_as_real(xc * rot).reshape(x.shape)

    out = torch.nn.functional.scaled_dot_product_attention(rotate(tq), rotate(tk), tv, is_causal=True,
                                                           enable_gqa=True)
    out.backward(tdo)
    np.testing.assert_allclose(dq[:, :, inv], tq.grad.numpy(), rtol=0, atol=2e-6)
    np.testing.assert_allclose(dk[:, :, inv], tk.grad.numpy(), rtol=0, atol=2e-6)


# ------------------------------------------------------------------------------------------------
# One device of the multi-device ring: the block functions
# ------------------------------------------------------------------------------------------------
def _shard(t, i, n):
    """Rows [i*S, (i+1)*S) of a [B, heads, L, d] (or [B, heads, L]) tensor: device i's local buffer."""
    S = t.shape[2] // n
    return t[:, :, i * S:(i + 1) * S].contiguous()


BLOCK_CASES = [  # B, H, Hkv, L, d, n, causal, layout
    (1, 2, 1, 32, 8, 4, True, "zigzag"),
    (2, 4, 2, 24, 8, 3, True, "contiguous"),
    (1, 2, 2, 32, 8, 4, True, "striped"),
    (1, 2, 1, 24, 8, 2, False, "zigzag"),
    (1, 1, 1, 16, 8, 1, True, "contiguous"),
]


@pytest.mark.parametrize("B,H,Hkv,L,d,n,causal,layout", BLOCK_CASES)
def test_block_fwd_blocks_recombine_into_full_attention(B, H, Hkv, L, d, n, causal, layout):
    """The n blocks a device meets partition its rows' key sets, so their (o_part, lse_part) merged by
    log-sum-exp weights give full attention (the pages: after n steps the ring result equals full
    attention).  Compared with the full-sequence oracle, which is pinned to torch's attention."""
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=torch.float32, seed=77 + L + n)
    ref_o, ref_l = oracle.attn_fwd(x["q"], x["k"], x["v"], n, causal, layout)
    for i in range(n):
        parts = [oracle.block_fwd(_shard(x["q"], i, n), _shard(x["k"], j, n), _shard(x["v"], j, n), L, n, causal,
                                  layout, i, j) for j in range(n)]
        lse = np.logaddexp.reduce(np.stack([p[1] for p in parts]), axis=0)
        o = sum(np.exp(p[1] - lse)[..., None] * p[0] for p in parts)
        S = L // n
        assert np.abs(lse - ref_l[:, :, i * S:(i + 1) * S]).max() < 1e-12
        assert np.abs(o - ref_o[:, :, i * S:(i + 1) * S]).max() < 1e-12


@pytest.mark.parametrize("layout", ["contiguous", "zigzag", "striped"])
def test_block_fwd_sees_exactly_the_ring_walks_pairs(layout):
    """With V the identity (d = S, v_t = e_t) the block output row shows which keys of the block the
    query saw; their count per (i, j) equals the visible pairs the oracle's ring walk counts at that
    step, which are pinned to closed forms elsewhere.  A block that sees nothing has lse = -inf, o = 0.
    This ties block (i, j) to the keys of shard j, not of another shard."""
    L, n = 32, 4
    S = L // n
    x = synth.make_inputs(1, 1, 1, L, S, dtype=torch.float32, seed=5)
    v = torch.eye(S).repeat(n, 1).view(1, 1, L, S)
    _, _, pairs = oracle.ring_fwd(x["q"], x["k"], v, n, True, layout)
    for i in range(n):
        for j in range(n):
            o, lse = oracle.block_fwd(_shard(x["q"], i, n), _shard(x["k"], j, n), _shard(v, j, n), L, n, True,
                                      layout, i, j)
            assert int((o > 0).sum()) == pairs[i, j]
            empty = np.isneginf(lse)
            assert np.all(o[empty] == 0)
            assert np.all((o > 0).sum(axis=-1)[~empty] > 0)


@pytest.mark.parametrize("B,H,Hkv,L,d,n,causal,layout", BLOCK_CASES)
def test_block_bwd_contributions_sum_to_the_full_gradients(B, H, Hkv, L, d, n, causal, layout):
    """Summed over the key shards j, a query shard's dq contributions are its rows of the full dq;
    summed over the query shards i, a key shard's dk and dv contributions are its rows of the full dk
    and dv (oracle_attn_bwd, pinned to torch autograd and finite differences)."""
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=torch.float32, seed=91 + L + n, with_dout=True)
    out, lse = oracle.attn_fwd(x["q"], x["k"], x["v"], n, causal, layout)
    D = (x["dout"].double().numpy() * out).sum(-1)
    rq, rk, rv = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], n, causal, layout)
    S = L // n
    dq = np.zeros_like(rq)
    dk = np.zeros_like(rk)
    dv = np.zeros_like(rv)
    for i in range(n):
        for j in range(n):
            a, b, c = oracle.block_bwd(_shard(x["q"], i, n), _shard(x["k"], j, n), _shard(x["v"], j, n),
                                       _shard(x["dout"], i, n), lse[:, :, i * S:(i + 1) * S],
                                       D[:, :, i * S:(i + 1) * S], L, n, causal, layout, i, j)
            dq[:, :, i * S:(i + 1) * S] += a
            dk[:, :, j * S:(j + 1) * S] += b
            dv[:, :, j * S:(j + 1) * S] += c
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert np.abs(got - ref).max() < 1e-11


def test_block_bwd_empty_block_is_zero():
    """Causal contiguous: keys of a later shard are never visible, so the block contributes nothing."""
    L, n = 24, 3
    x = synth.make_inputs(1, 2, 1, L, 8, dtype=torch.float32, seed=3, with_dout=True)
    lse = np.zeros((1, 2, 8))
    a, b, c = oracle.block_bwd(_shard(x["q"], 0, n), _shard(x["k"], 2, n), _shard(x["v"], 2, n),
                               _shard(x["dout"], 0, n), lse, lse, L, n, True, "contiguous", 0, 2)
    assert not a.any() and not b.any() and not c.any()
