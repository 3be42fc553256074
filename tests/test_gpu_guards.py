"""Out-of-bounds writes: every tensor a call receives sits inside a larger buffer whose margins (64 KB
on each side) hold a sentinel pattern; after the call the margins must be unchanged and the inputs
untouched.  Covers the fused forward and backward on both kernel paths (and their float32-output
forms), the per-device block calls,
the ring-step and stepwise forwards, RoPE and the Ulysses all-to-all (compute-sanitizer is not used
on this pool; this is its stand-in for writes)."""
import pytest
import torch

import sequence_sharded_exact_gb300 as ra
from sequence_sharded_exact_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
MARGIN = 64 * 1024  # bytes on each side


class Guarded:
    """Tensors carved out of one byte buffer, each between two sentinel margins."""

    def __init__(self):
        self.parts = []

    def new(self, shape, dtype, fill=None):
        nbytes = torch.empty(shape, dtype=dtype).numel() * torch.empty((), dtype=dtype).element_size()
        raw = torch.empty(2 * MARGIN + nbytes, dtype=torch.uint8, device=DEV)
        raw[:MARGIN] = 0xA5
        raw[MARGIN + nbytes:] = 0x5A
        t = raw[MARGIN:MARGIN + nbytes].view(dtype).view(shape)
        if fill is not None:
            t.copy_(fill)
        self.parts.append((raw, nbytes))
        return t

    def check(self):
        torch.cuda.synchronize()
        for raw, nbytes in self.parts:
            assert bool((raw[:MARGIN] == 0xA5).all()), "a write before a buffer"
            assert bool((raw[MARGIN + nbytes:] == 0x5A).all()), "a write after a buffer"


@pytest.fixture(autouse=True)
def _clean_status():
    torch.cuda.set_device(0)
    ra.device_status()
    yield
    assert ra.device_status() == 0


@pytest.mark.parametrize("B,H,Hkv,L,d,n,layout,dtype", [
    (1, 4, 2, 2048, 128, 4, "zigzag", torch.bfloat16),     # tensor-core paths
    (2, 2, 1, 1024, 64, 2, "striped", torch.bfloat16),
    (1, 2, 1, 768, 128, 3, "zigzag", torch.bfloat16),      # CUDA-core forward, tensor-core backward
    (1, 2, 2, 256, 64, 4, "contiguous", torch.float32),    # CUDA-core
])
def test_no_call_writes_outside_its_tensors(B, H, Hkv, L, d, n, layout, dtype):
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=dtype, seed=L + d, with_dout=True)
    g = Guarded()
    q, k, v, do = (g.new(x[t].shape, dtype, x[t].to(DEV)) for t in ("q", "k", "v", "dout"))
    keep = [t.clone() for t in (q, k, v, do)]
    out = g.new(q.shape, dtype)
    lse = g.new((B, H, L), torch.float32)
    ra.fwd(q, k, v, n, True, layout, out=out, lse=lse)
    g.check()
    for gd in (torch.float32, torch.bfloat16) if dtype == torch.bfloat16 else (torch.float32,):
        dq, dk, dv = g.new(q.shape, gd), g.new(k.shape, gd), g.new(v.shape, gd)
        ws = g.new((max(256, ra.bwd_workspace_size(B, H, Hkv, L, d, gd)),), torch.uint8)
        ra.bwd(q, k, v, out, lse, do, n, True, layout, grad_dtype=gd, dq=dq, dk=dk, dv=dv, workspace=ws)
        g.check()
    # the forward's float32 output and the backward that takes D from it
    o32, l32 = g.new(q.shape, torch.float32), g.new((B, H, L), torch.float32)
    ra.fwd_f32out(q, k, v, n, True, layout, out=o32, lse=l32)
    dq3, dk3, dv3 = g.new(q.shape, torch.float32), g.new(k.shape, torch.float32), g.new(v.shape, torch.float32)
    ws3 = g.new((max(256, ra.bwd_workspace_size(B, H, Hkv, L, d, torch.float32)),), torch.uint8)
    ra.bwd_f32out(q, k, v, o32, l32, do, n, True, layout, dq=dq3, dk=dk3, dv=dv3, workspace=ws3)
    g.check()
    # ring steps: a written partial, then a step folded into it; the stepwise forward
    op, lp = g.new((B, H, L, d), torch.float32), g.new((B, H, L), torch.float32)
    ra.ring_step_fwd(q, k, v, n, 0, True, layout, o_part=op, lse_part=lp)
    ra.ring_step_fwd_accumulate(q, k, v, n, n - 1, op, lp, True, layout)
    out2, lse2 = g.new(q.shape, dtype), g.new((B, H, L), torch.float32)
    ws2 = g.new((ra.library().ring_attn_fwd_stepwise_workspace_size(B, H, L, d),), torch.uint8)
    ra.fwd_stepwise(q, k, v, n, True, layout, out=out2, lse=lse2, workspace=ws2)
    g.check()
    # one device's block calls on local shard buffers
    S = L // n
    i, j = n - 1, 0
    sh = lambda t, s: t[:, :, s * S:(s + 1) * S].contiguous()
    qi, kj, vj, doi = (g.new(sh(t, s).shape, dtype, sh(t, s)) for t, s in ((q, i), (k, j), (v, j), (do, i)))
    ob, lb = g.new((B, H, S, d), torch.float32), g.new((B, H, S), torch.float32)
    ra.block_fwd(qi, kj, vj, ob, lb, n, i, j, False, True, layout)
    ra.block_fwd(qi, kj, vj, ob, lb, n, i, j, True, True, layout)
    Db = g.new((B, H, S), torch.float32, torch.zeros((B, H, S), device=DEV))
    dqa = g.new((B, H, S, d), torch.float32, torch.zeros((B, H, S, d), device=DEV))
    dkb, dvb = g.new((B, Hkv, S, d), torch.float32), g.new((B, Hkv, S, d), torch.float32)
    ra.block_bwd(qi, kj, vj, doi, lb, Db, dqa, dkb, dvb, n, i, j, False, True, layout)
    ra.block_bwd(qi, kj, vj, doi, lb, Db, dqa, dkb, dvb, n, i, j, True, True, layout)
    ra.bwd_preprocess(sh(out, i), doi, D=Db)
    ra.f32_add(dkb, dvb)
    ra.f32_convert(dqa, dtype, dst=g.new(dqa.shape, dtype))
    ra.block_rope(qi, n, i, layout)
    g.check()
    # RoPE in place and a Ulysses all-to-all, when the heads divide
    ra.rope(out, n, layout)
    if H % n == 0:
        tok = g.new((n, B, S, H, d), dtype, torch.randn((n, B, S, H, d), device=DEV).to(dtype))
        ra.ulysses_a2a(tok, n, layout, 0, dst=g.new((n, B, H // n, L, d), dtype))
    g.check()
    for a, b in zip(keep, (q, k, v, do)):
        assert torch.equal(a, b), "an input was written"
