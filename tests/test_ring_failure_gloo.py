"""Failure detection on the multi-device ring, on the host (gloo CPU ranks, no GPU): when a rank leaves
between steps or stops answering, its neighbours' transfers end with an error within the process
group's timeout (5 s here) and ring_fwd raises -- nobody waits for ever."""
import os
import time

import pytest
import torch.multiprocessing as mp

from ring_ranks import free_port, run_failing_rank


@pytest.mark.parametrize("mode", ["exit", "stall"])
def test_a_lost_rank_is_detected_by_its_neighbours(mode, tmp_path):
    world = 3
    ctx = mp.start_processes(run_failing_rank, args=(world, free_port(), mode, str(tmp_path)), nprocs=world,
                             join=False, start_method="spawn")
    t0 = time.time()
    survivors = [0, 2]
    while time.time() - t0 < 120:
        if all(os.path.exists(tmp_path / f"rank{r}.detected") or os.path.exists(tmp_path / f"rank{r}.err")
               for r in survivors):
            break
        time.sleep(0.5)
    for p in ctx.processes:  # the stalled rank (and anything left) is ended here
        if p.is_alive():
            p.kill()
        p.join(timeout=10)
    errs = [open(tmp_path / f"rank{r}.err").read() for r in survivors if os.path.exists(tmp_path / f"rank{r}.err")]
    assert not errs, errs
    # rank 2 receives from the lost rank 1 and must see the failure; rank 0 may too, or may block on
    # its own neighbour's failure in turn -- at least the neighbour that waits on rank 1 reports it
    detected = {r: open(tmp_path / f"rank{r}.detected").read() for r in survivors
                if os.path.exists(tmp_path / f"rank{r}.detected")}
    assert 2 in detected, f"rank 2 did not report the lost neighbour: {detected}"
    assert float(detected[2].split()[0]) < 60, detected
