"""Failure detection on the GPU without a fault: a bounded wait that nothing completes runs out,
reports through the device status word, and the context stays usable for attention."""
import pytest
import torch

import sequence_sharded_exact_gb300 as ra
from sequence_sharded_exact_gb300 import binding, synth

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports():
    torch.cuda.set_device(0)
    assert ra.device_status() == 0
    assert binding.selftest_bounded_wait(limit_ns=2_000_000) == 1       # the wait gave up after 2 ms
    assert ra.device_status() == binding.RA_DEVICE_TIMEOUT              # and said so
    assert ra.device_status() == 0                                      # reading clears the word
    # the same report as a status code: ring_attn_device_check returns RA_ERR_TIMEOUT, then RA_OK
    assert binding.selftest_bounded_wait(limit_ns=2_000_000) == 1
    with pytest.raises(binding.RingAttnError) as err:
        ra.device_check()
    assert err.value.status == binding.RA_ERR_TIMEOUT and "bounded wait" in str(err.value)
    ra.device_check()                                                   # the word was cleared
    # the context is intact: a forward still runs and the status stays clean
    x = synth.make_inputs(1, 2, 1, 1024, 128, dtype=torch.bfloat16, seed=5, device="cuda:0")
    out, lse = ra.fwd(x["q"], x["k"], x["v"], 4, True, "zigzag")
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and ra.device_status() == 0
