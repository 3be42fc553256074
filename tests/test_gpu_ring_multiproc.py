"""The multi-device ring through the library's block kernels, with its ranks as separate processes
that share cuda:0 and pass the blocks over gloo (staged through host memory).  No kernel waits on
another rank: every exchange happens on the host between launches, so the ranks' kernels are
independent launches.  Each rank checks its shard of out, lse, dq, dk and dv against the float64
oracle of the whole sequence, in the contiguous, zigzag and striped layouts, on the tensor-core
path (bf16, head dim 128 and 64) and on the CUDA-core path (float32); two cases rotate q and k by
natural position on each rank first (ring_attn_block_rope), as the pages ask when blocks travel."""
import pytest
import torch

from ring_ranks import launch, precompute_refs

pytestmark = pytest.mark.gpu

CASES = {  # B, H, Hkv, L, d, causal, layout, dtype, grad dtype, seed
    2: [(1, 4, 2, 4096, 128, True, "zigzag", "bfloat16", "float32", 201),
        (1, 2, 1, 2048, 128, True, "contiguous", "bfloat16", "bfloat16", 202),
        (1, 2, 2, 2048, 64, True, "striped", "bfloat16", "float32", 203),
        (1, 2, 1, 512, 64, True, "zigzag", "float32", "float32", 204),
        (1, 4, 2, 4096, 128, True, "zigzag", "bfloat16", "float32", 210, 10000.0)],  # RoPE by natural position
    4: [(1, 4, 2, 4096, 128, True, "zigzag", "bfloat16", "float32", 205),
        (2, 2, 1, 2048, 128, True, "contiguous", "bfloat16", "float32", 206),
        (1, 4, 1, 4096, 128, True, "striped", "bfloat16", "float32", 207),
        (1, 2, 1, 2048, 128, False, "zigzag", "bfloat16", "float32", 208),
        (1, 2, 2, 512, 128, True, "zigzag", "float32", "float32", 209),
        (1, 2, 1, 4096, 128, True, "striped", "bfloat16", "float32", 211, 500000.0)],
}


@pytest.mark.parametrize("world", [2, 4])
def test_ring_processes_on_one_gpu_match_the_oracle(world, tmp_path):
    assert torch.cuda.is_available()
    precompute_refs(world, CASES[world], str(tmp_path))
    ok, errs = launch(world, CASES[world], "cuda", str(tmp_path), timeout=900)
    assert ok, "\n".join(errs)


def test_hierarchical_ring_processes_on_one_gpu_match_the_oracle(tmp_path):
    """The hierarchical ring over 4 ranks in 2 groups of 2 (local ring inside a group, global ring
    across the groups), through the library's kernels."""
    cases = [CASES[4][0], CASES[4][2], CASES[4][4]]
    precompute_refs(4, cases, str(tmp_path))
    ok, errs = launch(4, cases, "cuda", str(tmp_path), timeout=900, groups=2)
    assert ok, "\n".join(errs)


@pytest.mark.parametrize("groups", [1, 2])
def test_distributed_ring_attention_autograd_on_one_gpu(groups, tmp_path):
    """ring_attention_distributed with the library's kernels: 4 ranks (flat, or 2 groups of 2) share
    cuda:0; forward and autograd gradients (bf16) of every rank against the oracle."""
    import os
    import torch.multiprocessing as mp

    from ring_ranks import free_port, run_autograd_rank

    mp.start_processes(run_autograd_rank, args=(4, free_port(), groups, str(tmp_path), "cuda"), nprocs=4,
                       join=True, start_method="spawn")
    errs = [open(tmp_path / f"rank{r}.err").read() for r in range(4) if os.path.exists(tmp_path / f"rank{r}.err")]
    assert not errs, "\n".join(errs)


def test_pages_ring_attention_object_on_one_gpu(tmp_path):
    """RingAttention(dim, heads, rank, world_size) with its defaults (no mask, contiguous shards) on
    the library's kernels: 2 ranks share cuda:0; forward and gradients against the oracle."""
    import os
    import torch.multiprocessing as mp

    from ring_ranks import free_port, run_autograd_rank

    mp.start_processes(run_autograd_rank, args=(2, free_port(), 1, str(tmp_path), "cuda", False, "contiguous", True),
                       nprocs=2, join=True, start_method="spawn")
    errs = [open(tmp_path / f"rank{r}.err").read() for r in range(2) if os.path.exists(tmp_path / f"rank{r}.err")]
    assert not errs, "\n".join(errs)
    assert all(os.path.exists(tmp_path / f"rank{r}.ok") for r in range(2))


@pytest.mark.parametrize("step", ["fwd", "train"])
def test_bench_ring_mode_with_two_ranks(step):
    """bench.py's multi-rank ring mode, as a launcher runs it for N > 1 (here 2 gloo ranks sharing
    cuda:0 instead of NCCL across 2 GPUs): one JSON line from rank 0, alone on stdout, with the whole
    sequence's TFLOP/s, a clean status word, the roofline of the block launches and the end-to-end
    leg."""
    import json
    import pathlib
    import subprocess
    import sys

    from ring_ranks import free_port

    root = pathlib.Path(__file__).resolve().parents[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py", "--gpus", "2",
           "--steps", "2", "--warmup", "3", "--workload", "zigzag_gqa_32k", "--step", step,
           "--dist-backend", "gloo"]
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    printed = [x for x in r.stdout.splitlines() if x.strip()]
    assert len(printed) == 1, r.stdout  # the JSON line and nothing else on stdout
    lines = [json.loads(printed[0])]
    line = lines[0]
    assert line["n_gpus"] == 2 and line["steps"] == 2 and line["scaling"] == "strong"
    assert line["device_status"] == 0 and line["value"] > 0 and line["ms_per_step"] > 0
    assert line["config"]["n_shards"] == 2 and "GLOO" in line["config"]["mode"]
    assert 0 < line["roofline"]["frac"] < 1.5
    # the two ranks together copy in every row of q, k, v (and dO), bf16, and copy out every row of
    # out (bf16) and lse (float32)
    L, H, Hkv, d = 32768, 32, 8, 128
    h2d = 2 * L * d * (H + 2 * Hkv) + (2 * L * d * H if step == "train" else 0)
    assert line["e2e"]["h2d_bytes_per_step"] == h2d
    assert line["e2e"]["d2h_bytes_per_step"] == 2 * L * d * H + 4 * L * H
    assert line["e2e"]["value"] > 0


def test_eight_ranks_at_16k_flat_and_hierarchical(tmp_path):
    """Eight ranks (processes sharing cuda:0) on a 16384-token zigzag sequence, 8 query heads on 2 kv
    heads: the flat ring, then the hierarchical ring in 2 groups of 4; every rank's shard of out,
    lse, dq, dk and dv against the float64 oracle of the whole sequence (computed once)."""
    import os

    case = (1, 8, 2, 16384, 128, True, "zigzag", "bfloat16", "float32", 212)
    precompute_refs(8, [case], str(tmp_path))
    for groups in (None, 2):
        for r in range(8):
            for suffix in ("ok", "err"):
                f = tmp_path / f"rank{r}.{suffix}"
                if os.path.exists(f):
                    os.remove(f)
        ok, errs = launch(8, [case], "cuda", str(tmp_path), timeout=900, groups=groups)
        assert ok, f"groups={groups}:\n" + "\n".join(errs)


def test_distributed_ring_attention_keeping_the_float32_output_on_one_gpu(tmp_path):
    """ring_attention_distributed(..., f32_out=True) with the library's kernels, 4 ranks sharing
    cuda:0: the backward's D from each rank's float32 running output (the mixed-precision
    preprocess); forward and gradients against the oracle."""
    import os
    import torch.multiprocessing as mp

    from ring_ranks import free_port, run_autograd_rank

    mp.start_processes(run_autograd_rank, args=(4, free_port(), 1, str(tmp_path), "cuda", True, "zigzag", False, True),
                       nprocs=4, join=True, start_method="spawn")
    errs = [open(tmp_path / f"rank{r}.err").read() for r in range(4) if os.path.exists(tmp_path / f"rank{r}.err")]
    assert not errs, "\n".join(errs)
    assert all(os.path.exists(tmp_path / f"rank{r}.ok") for r in range(4))
