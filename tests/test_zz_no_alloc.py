"""ring_attn_bwd_static_scratch: the backward for callers that cannot allocate device memory (a host
framework that owns all device memory as one pool and hands over only input and output buffers,
or a loop that may not call the allocator).  Its scratch is a fixed device array inside the
library.  These tests call it through the C ABI and compare it with ring_attn_bwd, which takes a
caller workspace, on two calls in a row (the second call must not see the first call's leftovers).
"""
import ctypes

import pytest
import torch

import sequence_sharded_exact_gb300 as ra
from sequence_sharded_exact_gb300 import binding, synth
from parity_util import assert_close, to_np


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


@pytest.mark.gpu
def test_static_scratch_backward_matches_workspace_backward_twice():
    torch.cuda.set_device(0)
    dev = "cuda:0"
    calls = [
        # (B, H, Hkv, L, n, layout, grad dtype, seed): tensor-core path, the scratch holds D and
        # the float32 dQ accumulator
        (1, 4, 2, 2048, 4, "zigzag", torch.bfloat16, 31),
        # a smaller problem next: what the first call left in the scratch must not leak in
        (1, 2, 1, 1024, 2, "contiguous", torch.bfloat16, 32),
    ]
    for B, H, Hkv, L, n, layout, gdt, seed in calls:
        x = synth.make_inputs(B, H, Hkv, L, 128, dtype=torch.bfloat16, seed=seed, with_dout=True)
        q, k, v, do = (x[t].to(dev) for t in ("q", "k", "v", "dout"))
        out, lse = ra.fwd(q, k, v, n, True, layout)
        ref = ra.bwd(q, k, v, out, lse, do, n, True, layout, grad_dtype=gdt)
        got = binding.bwd_static_scratch(q, k, v, out, lse, do, n, True, layout, grad_dtype=gdt)
        torch.cuda.synchronize()
        assert ra.device_status() == 0
        for g, r, name in zip(got, ref, ("dq", "dk", "dv")):
            assert g.dtype == gdt
            assert_close(to_np(g), to_np(r), torch.bfloat16, name, stored_bf16=True)
