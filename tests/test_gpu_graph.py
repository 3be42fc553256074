"""The library's calls inside a CUDA graph: after one ordinary call (which sets the kernels' launch
attributes and looks up the device status word), a forward and a backward are captured with
torch.cuda.graph and replayed on new inputs written into the same buffers; the replay gives the
results of ordinary calls on those inputs.  Only kernel launches are enqueued, so the calls record
into a graph like any stream work: a step that repeats with the same shapes can be launched as one
graph."""
import pytest
import torch

import sequence_sharded_exact_gb300 as ra
from sequence_sharded_exact_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("B,H,Hkv,L,d,n,layout,dtype", [
    (1, 4, 2, 2048, 128, 4, "zigzag", torch.bfloat16),   # tensor-core kernels
    (1, 2, 1, 768, 64, 3, "striped", torch.float32),     # CUDA-core kernels
])
def test_forward_and_backward_replayed_from_a_cuda_graph(B, H, Hkv, L, d, n, layout, dtype):
    torch.cuda.set_device(0)
    ra.device_status()
    a = synth.make_inputs(B, H, Hkv, L, d, dtype=dtype, seed=71, with_dout=True)
    b = synth.make_inputs(B, H, Hkv, L, d, dtype=dtype, seed=72, with_dout=True)
    q, k, v, do = (a[t].to(DEV) for t in ("q", "k", "v", "dout"))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=DEV)
    dq = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    dk = torch.empty(k.shape, dtype=torch.float32, device=DEV)
    dv = torch.empty(v.shape, dtype=torch.float32, device=DEV)
    ws = torch.empty(max(256, ra.bwd_workspace_size(B, H, Hkv, L, d, torch.float32)), dtype=torch.uint8,
                     device=DEV)

    def step():
        ra.fwd(q, k, v, n, True, layout, out=out, lse=lse)
        ra.bwd(q, k, v, out, lse, do, n, True, layout, dq=dq, dk=dk, dv=dv, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # ordinary calls first
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for t, src in ((q, b["q"]), (k, b["k"]), (v, b["v"]), (do, b["dout"])):
        t.copy_(src.to(DEV))
    graph.replay()
    torch.cuda.synchronize()
    assert ra.device_status() == 0
    ref_o, ref_l = ra.fwd(q, k, v, n, True, layout)
    ref_q, ref_k, ref_v = ra.bwd(q, k, v, ref_o, ref_l, do, n, True, layout)
    torch.cuda.synchronize()
    # the forward and dK, dV add in a fixed order: the same bits; dQ is summed with atomics in
    # arrival order, which can move the last bits of a float32 sum
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    assert torch.equal(dk, ref_k) and torch.equal(dv, ref_v)
    assert torch.allclose(dq, ref_q, rtol=1e-5, atol=1e-5)
    # and the graph computed the new inputs' results, not the first ones'
    old_o, _ = ra.fwd(a["q"].to(DEV), a["k"].to(DEV), a["v"].to(DEV), n, True, layout)
    assert not torch.equal(out, old_o)
