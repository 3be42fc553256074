"""Seeded synthetic inputs for Ring Attention workloads.

This module draws random tensors and nothing else: it holds none of the attention arithmetic, so
that the CUDA path and the float64 oracle can both be fed from it without sharing any of the method.

Recipe (the same for every workload):
  * q [B,H,L,d], k and v [B,Hkv,L,d] and, for the backward, dout [B,H,L,d] are i.i.d. N(0,1)
    drawn in float32 from a seeded generator, in that order;
  * optionally a fraction of key rows is multiplied by a factor (the long-context workload scales
    round(0.01 * L) seeded rows of every (batch, kv head) by 8, stressing the running maximum);
  * the tensors are then rounded to the compute dtype (round-to-nearest-even for bf16); the oracle
    reads exactly these rounded values.
The rows are drawn in buffer order; since they are i.i.d. the layout does not change their law.
"""
from __future__ import annotations

import torch

# The workloads of the benchmark and parity suite (sizes as quoted on the pages' examples: 128K
# tokens over 8 shards of 16K, head dim 128, inner tile 128).  The striped ones repeat the zigzag
# sizes in the round-robin layout, the _d64 ones with head dim 64.
WORKLOADS = {
    "tiny_f32": dict(B=1, H=1, Hkv=1, L=256, d=64, n=4, causal=False, layout="contiguous",
                     dtype=torch.float32, spike_frac=0.0, backward=False, seed=1001),
    "causal_contig_8k": dict(B=2, H=8, Hkv=8, L=8192, d=128, n=8, causal=True, layout="contiguous",
                             dtype=torch.bfloat16, spike_frac=0.0, backward=False, seed=1002),
    "zigzag_gqa_32k": dict(B=1, H=32, Hkv=8, L=32768, d=128, n=8, causal=True, layout="zigzag",
                           dtype=torch.bfloat16, spike_frac=0.0, backward=False, seed=1003),
    "zigzag_gqa_128k": dict(B=1, H=32, Hkv=8, L=131072, d=128, n=8, causal=True, layout="zigzag",
                            dtype=torch.bfloat16, spike_frac=0.01, backward=False, seed=1004),
    "zigzag_gqa_64k_train": dict(B=1, H=32, Hkv=8, L=65536, d=128, n=16, causal=True,
                                 layout="zigzag", dtype=torch.bfloat16, spike_frac=0.0,
                                 backward=True, seed=1005),
    "striped_gqa_128k": dict(B=1, H=32, Hkv=8, L=131072, d=128, n=8, causal=True, layout="striped",
                             dtype=torch.bfloat16, spike_frac=0.01, backward=False, seed=1006),
    "striped_gqa_64k_train": dict(B=1, H=32, Hkv=8, L=65536, d=128, n=16, causal=True,
                                  layout="striped", dtype=torch.bfloat16, spike_frac=0.0,
                                  backward=True, seed=1007),
    # head dim 64 (the other head dim of the tensor-core kernels), same sequences
    "zigzag_gqa_128k_d64": dict(B=1, H=32, Hkv=8, L=131072, d=64, n=8, causal=True, layout="zigzag",
                                dtype=torch.bfloat16, spike_frac=0.01, backward=False, seed=1008),
    "zigzag_gqa_64k_train_d64": dict(B=1, H=32, Hkv=8, L=65536, d=64, n=16, causal=True,
                                     layout="zigzag", dtype=torch.bfloat16, spike_frac=0.0,
                                     backward=True, seed=1009),
}


def make_inputs(B, H, Hkv, L, d, dtype=torch.bfloat16, seed=0, spike_frac=0.0, spike_scale=8.0,
                with_dout=False, device="cpu", gen_device="cpu"):
    """Return a dict with q, k, v (and dout) on `device`, already rounded to `dtype`.

    The draw happens on the generator of `gen_device` ("cpu" by default, so that the values do
    not depend on where they are used; "cuda" draws the large workloads quickly, from the device's
    own generator stream)."""
    g = torch.Generator(device=gen_device)
    g.manual_seed(int(seed))
    f32 = dict(generator=g, dtype=torch.float32, device=gen_device)
    q = torch.randn((B, H, L, d), **f32)
    k = torch.randn((B, Hkv, L, d), **f32)
    v = torch.randn((B, Hkv, L, d), **f32)
    dout = torch.randn((B, H, L, d), **f32) if with_dout else None
    if spike_frac > 0.0:
        count = int(round(spike_frac * L))
        for bh in range(B * Hkv):
            rows = torch.randperm(L, generator=g, device=gen_device)[:count]
            k.view(B * Hkv, L, d)[bh, rows] *= spike_scale
    out = {"q": q, "k": k, "v": v}
    if dout is not None:
        out["dout"] = dout
    res = {}
    for name in list(out):
        res[name] = out.pop(name).to(dtype).to(device)
    return res


def make_workload(name, device="cpu", with_dout=None, gen_device="cpu"):
    w = WORKLOADS[name]
    wd = w["backward"] if with_dout is None else with_dout
    return make_inputs(w["B"], w["H"], w["Hkv"], w["L"], w["d"], dtype=w["dtype"], seed=w["seed"],
                       spike_frac=w["spike_frac"], with_dout=wd, device=device,
                       gen_device=gen_device)
