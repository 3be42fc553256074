"""The multi-device ring on CPU ranks (gloo, world sizes 2 to 4): sequence_sharded_exact_gb300.ring
schedules the blocks and moves them with torch.distributed point-to-point operations, and the
per-device compute is the float64 oracle's block functions (world size 1 is the degenerate ring: one
device, one block, no transfer).  Every rank checks its shard of out,
lse, dq, dk and dv against the oracle of the whole sequence (1e-10), and the order of its block calls
(step r computes block (rank - r) mod n; the first writes, the later ones fold in)."""
import pytest

from ring_ranks import launch

CASES = [  # B, H, Hkv, L, d, causal, layout, dtype, grad dtype, seed
    (1, 2, 1, 48, 8, True, "zigzag", "float32", "float32", 11),
    (1, 2, 2, 48, 8, True, "contiguous", "float32", "float32", 12),
    (2, 2, 1, 48, 8, True, "striped", "float32", "float32", 13),
    (1, 2, 1, 48, 8, False, "zigzag", "float32", "float32", 14),
]


@pytest.mark.parametrize("world", [1, 2, 3, 4])
def test_ring_on_gloo_ranks_matches_full_attention(world, tmp_path):
    cases = [c for c in CASES if c[3] % (2 * world) == 0]
    ok, errs = launch(world, cases, "cpu", str(tmp_path), timeout=300)
    assert ok, "\n".join(errs)


@pytest.mark.parametrize("world,groups", [(4, 2), (6, 2), (6, 3), (3, 1), (3, 3), (8, 4)])
def test_hierarchical_ring_on_gloo_ranks_matches_full_attention(world, groups, tmp_path):
    """The hierarchical ring (local ring inside groups of world / groups ranks, global ring across
    them): same results as the flat ring, every shard met once, accumulators home at the end."""
    cases = [c for c in CASES if c[3] % (2 * world) == 0] or [(1, 2, 1, 96, 8, True, "zigzag", "float32",
                                                                 "float32", 15)]
    ok, errs = launch(world, cases, "cpu", str(tmp_path), timeout=300, groups=groups)
    assert ok, "\n".join(errs)


@pytest.mark.parametrize("world,groups", [(2, 1), (4, 2)])
def test_distributed_ring_attention_under_autograd(world, groups, tmp_path):
    """ring_attention_distributed: the forward and the gradients autograd produces on every rank are
    that rank's shard of the whole-sequence oracle (flat and hierarchical ring)."""
    import os
    import torch.multiprocessing as mp

    from ring_ranks import free_port, run_autograd_rank

    mp.start_processes(run_autograd_rank, args=(world, free_port(), groups, str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    errs = [open(tmp_path / f"rank{r}.err").read() for r in range(world) if os.path.exists(tmp_path / f"rank{r}.err")]
    assert not errs, "\n".join(errs)
    assert all(os.path.exists(tmp_path / f"rank{r}.ok") for r in range(world))


@pytest.mark.parametrize("world,groups,causal,layout", [(3, 1, False, "contiguous"), (4, 2, True, "striped")])
def test_pages_ring_attention_object(world, groups, causal, layout, tmp_path):
    """RingAttention(dim, heads, rank, world_size), the pages' per-rank object (no mask and contiguous
    shards by default): forward and autograd gradients on every rank equal its shard of the oracle;
    a rank or world size that disagrees with the process group, and a q whose head dim is not
    dim // heads, are refused."""
    import os
    import torch.multiprocessing as mp

    from ring_ranks import free_port, run_autograd_rank

    mp.start_processes(run_autograd_rank, args=(world, free_port(), groups, str(tmp_path), "cpu", causal, layout, True),
                       nprocs=world, join=True, start_method="spawn")
    errs = [open(tmp_path / f"rank{r}.err").read() for r in range(world) if os.path.exists(tmp_path / f"rank{r}.err")]
    assert not errs, "\n".join(errs)
    assert all(os.path.exists(tmp_path / f"rank{r}.ok") for r in range(world))


def test_distributed_ring_attention_keeping_the_float32_output(tmp_path):
    """ring_attention_distributed(..., f32_out=True): the backward takes D from the forward's running
    output (the plumbing of the float32 output through the autograd function), 3 gloo CPU ranks."""
    import os
    import torch.multiprocessing as mp

    from ring_ranks import free_port, run_autograd_rank

    mp.start_processes(run_autograd_rank, args=(3, free_port(), 1, str(tmp_path), "cpu", True, "zigzag", False, True),
                       nprocs=3, join=True, start_method="spawn")
    errs = [open(tmp_path / f"rank{r}.err").read() for r in range(3) if os.path.exists(tmp_path / f"rank{r}.err")]
    assert not errs, "\n".join(errs)
    assert all(os.path.exists(tmp_path / f"rank{r}.ok") for r in range(3))
