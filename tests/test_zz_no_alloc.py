"""ring_attn_bwd_static_scratch: the backward for callers that cannot allocate device memory (a host
framework that owns all device memory as one pool and hands over only input and output buffers,
or a loop that may not call the allocator).  Its scratch is a fixed device array inside the
library.  These tests call it through the C ABI and compare it with ring_attn_bwd, which takes a
caller workspace, on calls in a row (a later call must not see an earlier call's leftovers), with
both gradient dtypes: bf16 gradients keep the row sums and the float32 dQ accumulator in the
scratch, float32 gradients keep only the row sums there and accumulate dQ in the caller's buffer.

The two paths run the same kernels, so they are compared with each other far more tightly than
with the oracle: dK and dV come from one CTA each in a fixed order and must agree bit for bit;
dQ is summed with floating-point atomics in whatever order the CTAs arrive, so it may differ by
float32 reordering (and, stored in bf16, by one bf16 rounding step of the value).
"""
import ctypes

import numpy as np
import pytest
import torch

import sequence_sharded_exact_gb300 as ra
from sequence_sharded_exact_gb300 import binding, synth
from parity_util import errors, to_np


def test_capacity_and_rejection_beyond_it():
    """Problems whose scratch would exceed the array are refused before anything runs."""
    cap = binding.bwd_static_scratch_capacity()
    assert cap == 64 << 20
    lib = binding.library()
    P = ctypes.c_void_p
    # bf16 gradients need 4 * (d + 1) bytes per query row: 4 heads x 131072 rows is ~270 MB
    st = lib.ring_attn_bwd_static_scratch(P(16), P(16), P(16), P(16), P(16), P(16), P(16), P(16),
                                          P(16), 1, 1, 4, 1, 131072, 128, 8, 1, 1, 1, None)
    assert st == binding.RA_ERR_INVALID_ARG
    assert "static scratch" in lib.ring_attn_last_error().decode()


def _assert_same_dq(got, ref, gdt):
    g, r = to_np(got), to_np(ref)
    if gdt == torch.float32:
        ma, rl = errors(g, r)
        assert ma <= 1e-4 and rl <= 1e-5, f"dq: max-abs {ma:.3e}, rel-L2 {rl:.3e}"
    else:
        # float32 sums that differ in their last bits can round to neighbouring bf16 values:
        # at most one bf16 step (2^-7 |x| relative, plus a float32-sized absolute slack)
        excess = np.abs(g - r) - (np.abs(r) * 2.0 ** -7 + 1e-6)
        assert float(excess.max()) <= 0, f"dq: differs by more than one bf16 step ({excess.max():.3e})"
        _, rl = errors(g, r)
        assert rl <= 1e-3, f"dq: rel-L2 {rl:.3e}"


@pytest.mark.gpu
def test_static_scratch_backward_matches_workspace_backward_twice():
    torch.cuda.set_device(0)
    dev = "cuda:0"
    calls = [
        # (B, H, Hkv, L, n, layout, grad dtype, seed), all on the tensor-core path
        (1, 4, 2, 2048, 4, "zigzag", torch.bfloat16, 31),   # scratch: D + float32 dQ accumulator
        (1, 2, 1, 1024, 2, "contiguous", torch.bfloat16, 32),  # smaller: no leftovers may leak in
        (1, 4, 2, 2048, 4, "zigzag", torch.float32, 33),    # scratch: D only; dQ accumulates in dq
        (2, 2, 2, 1024, 2, "striped", torch.float32, 34),
    ]
    for B, H, Hkv, L, n, layout, gdt, seed in calls:
        x = synth.make_inputs(B, H, Hkv, L, 128, dtype=torch.bfloat16, seed=seed, with_dout=True)
        q, k, v, do = (x[t].to(dev) for t in ("q", "k", "v", "dout"))
        out, lse = ra.fwd(q, k, v, n, True, layout)
        ref = ra.bwd(q, k, v, out, lse, do, n, True, layout, grad_dtype=gdt)
        got = binding.bwd_static_scratch(q, k, v, out, lse, do, n, True, layout, grad_dtype=gdt)
        torch.cuda.synchronize()
        assert ra.device_status() == 0
        for g in got:
            assert g.dtype == gdt and torch.isfinite(g.float()).all()
        _assert_same_dq(got[0], ref[0], gdt)
        assert torch.equal(got[1], ref[1]), "dk differs"
        assert torch.equal(got[2], ref[2]), "dv differs"
