"""The binding checks every tensor (device, contiguity, shape, dtype) before a pointer reaches the
library, which trusts the sizes it is given: a wrong tensor is an exception, never a launch."""
import pytest
import torch

import sequence_sharded_exact_gb300 as ra

B, H, Hkv, L, d, n = 1, 4, 2, 512, 64, 2


def _cpu(*shape, dtype=torch.bfloat16):
    return torch.zeros(shape, dtype=dtype)


def _calls(q, k, v, o, lse, do, f32o, f32l, ws):
    """Every tensor-taking entry point, called with the given tensors."""
    return {
        "fwd": lambda: ra.fwd(q, k, v, n),
        "fwd_tile_visits": lambda: ra.fwd_tile_visits(q, k, v, n),
        "ring_step_fwd": lambda: ra.ring_step_fwd(q, k, v, n, 0),
        "ring_step_fwd_accumulate": lambda: ra.ring_step_fwd_accumulate(q, k, v, n, 0, f32o, f32l),
        "lse_merge": lambda: ra.lse_merge(f32o, f32l, f32o.clone(), f32l.clone()),
        "fwd_stepwise": lambda: ra.fwd_stepwise(q, k, v, n, workspace=ws),
        "bwd": lambda: ra.bwd(q, k, v, o, lse, do, n, workspace=ws),
        "bwd_tile_visits": lambda: ra.bwd_tile_visits(q, k, v, o, lse, do, n),
        "bwd_static_scratch": lambda: ra.bwd_static_scratch(q, k, v, o, lse, do, n),
        "rope": lambda: ra.rope(q, n),
    }


def test_host_tensors_are_refused_before_any_launch():
    q, k, v = _cpu(B, H, L, d), _cpu(B, Hkv, L, d), _cpu(B, Hkv, L, d)
    o, do = _cpu(B, H, L, d), _cpu(B, H, L, d)
    lse = _cpu(B, H, L, dtype=torch.float32)
    f32o, f32l = _cpu(B, H, L, d, dtype=torch.float32), _cpu(B, H, L, dtype=torch.float32)
    ws = torch.zeros(1 << 20, dtype=torch.uint8)
    for name, call in _calls(q, k, v, o, lse, do, f32o, f32l, ws).items():
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()
    tq = _cpu(n, B, L // n, H, d)
    tk = _cpu(n, B, L // n, Hkv, d)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ra.ulysses_fwd(tq, tk, tk.clone(), n)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ra.ulysses_bwd(tq, tk, tk.clone(), tq.clone(), _cpu(n, B, L // n, H, dtype=torch.float32),
                       tq.clone(), n)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ra.ulysses_a2a(tq, n)


def test_host_buffer_forward_checks_shapes_and_dtypes():
    q, k = _cpu(B, H, L, d), _cpu(B, Hkv, L, d)
    out, lse = _cpu(B, H, L, d), _cpu(B, H, L, dtype=torch.float32)
    with pytest.raises(ValueError, match="shape"):
        ra.fwd_host(q, k, _cpu(B, Hkv, L - 2, d), n, out=out, lse=lse, device="cuda:0")
    with pytest.raises(ValueError, match="shape"):
        ra.fwd_host(q, k, k.float(), n, out=out, lse=lse, device="cuda:0")
    with pytest.raises(ValueError, match="contiguous CPU"):
        ra.fwd_host(q, k, k.transpose(2, 3).contiguous().transpose(2, 3), n, out=out, lse=lse,
                    device="cuda:0")


@pytest.mark.gpu
def test_device_tensors_with_wrong_sizes_are_refused():
    dev = "cuda:0"
    z = lambda *s, dtype=torch.bfloat16: torch.zeros(s, dtype=dtype, device=dev)  # noqa: E731
    q, k, v = z(B, H, L, d), z(B, Hkv, L, d), z(B, Hkv, L, d)
    o, do, lse = z(B, H, L, d), z(B, H, L, d), z(B, H, L, dtype=torch.float32)
    ra.device_status()
    bad = {
        "short k": dict(k=z(B, Hkv, L // 2, d)),
        "wider v": dict(v=z(B, Hkv, L, 2 * d)),
        "f32 v": dict(v=z(B, Hkv, L, d, dtype=torch.float32)),
        "strided k": dict(k=z(B, Hkv, d, L).transpose(2, 3)),
        "short out": dict(o=z(B, H, L - 128, d)),
        "bf16 lse": dict(lse=z(B, H, L)),
        "short dout": dict(do=z(B, H, L // 2, d)),
    }
    for what, repl in bad.items():
        t = dict(q=q, k=k, v=v, o=o, lse=lse, do=do)
        t.update(repl)
        uses_out = what in ("short out", "bf16 lse", "short dout")
        with pytest.raises(ValueError):
            if uses_out:
                ra.bwd(t["q"], t["k"], t["v"], t["o"], t["lse"], t["do"], n)
            else:
                ra.fwd(t["q"], t["k"], t["v"], n)
    with pytest.raises(ValueError):
        ra.bwd(q, k, v, o, lse, do, n, dq=z(B, H, L, d, dtype=torch.float32)[:, :, :-1])
    with pytest.raises(ValueError):
        ra.bwd(q, k, v, o, lse, do, n, workspace=torch.zeros(64, dtype=torch.uint8, device=dev))
    with pytest.raises(ValueError):
        ra.ring_step_fwd(q, k, v, n, 0, o_part=z(B, H, L, d))  # bf16 partial
    torch.cuda.synchronize()
    assert ra.device_status() == 0
