"""Worker side of the multi-process ring tests (spawned ranks; imported by the test modules).

Each rank builds the same seeded whole-sequence inputs, keeps its own shard, runs the ring forward
and backward through sequence_sharded_exact_gb300.ring with torch.distributed (gloo) moving the
blocks, and checks its shard of the results against the float64 oracle of the whole sequence."""
import os
import socket
import sys
import traceback

import numpy as np
import torch
import torch.distributed as dist

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def shard(t, i, n):
    S = t.shape[2] // n
    return t[:, :, i * S:(i + 1) * S].contiguous()


class OracleOps:
    """The ring's per-device compute done by the float64 oracle's block functions (CPU), so that the
    driver's schedule and transfers can be checked on CPU ranks.  Records every block call."""

    def __init__(self, L):
        import oracle

        self.oracle = oracle
        self.L = L
        self.calls = []

    def empty_acc(self, shape, like):
        return torch.empty(shape, dtype=torch.float64)

    def block_fwd(self, q, k, v, o_acc, lse_acc, n, i, j, accumulate, causal, layout):
        self.calls.append(("fwd", i, j, bool(accumulate)))
        o, l = self.oracle.block_fwd(q, k, v, self.L, n, causal, layout, i, j)
        o, l = torch.from_numpy(o), torch.from_numpy(l)
        if not accumulate:
            o_acc.copy_(o)
            lse_acc.copy_(l)
            return
        new = torch.logaddexp(lse_acc, l)
        keep = torch.isneginf(new)
        wa = torch.where(keep, torch.zeros_like(new), torch.exp(lse_acc - new))
        wb = torch.where(keep, torch.zeros_like(new), torch.exp(l - new))
        o_acc.copy_(wa[..., None] * o_acc + wb[..., None] * o)
        lse_acc.copy_(torch.where(keep, lse_acc, new))

    def convert(self, src, dtype):
        return src.clone()

    def preprocess(self, out, dout):
        return (out.double() * dout.double()).sum(-1)

    def zero(self, x):
        x.zero_()

    def block_bwd(self, q, k, v, dout, lse, D, dq_acc, dk, dv, n, i, j, accumulate_kv, causal, layout):
        self.calls.append(("bwd", i, j, bool(accumulate_kv)))
        a, b, c = self.oracle.block_bwd(q, k, v, dout, lse, D, self.L, n, causal, layout, i, j)
        dq_acc += torch.from_numpy(a)
        if accumulate_kv:
            dk += torch.from_numpy(b)
            dv += torch.from_numpy(c)
        else:
            dk.copy_(torch.from_numpy(b))
            dv.copy_(torch.from_numpy(c))

    def add(self, acc, part):
        acc += part


def errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    ma = float(np.abs(got - ref).max())
    rl = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    return ma, rl


def reference(x, n, causal, layout, rope_base):
    """The float64 oracle of the whole sequence: out, lse and the gradients with respect to q, k, v.
    With rope_base, q and k are first rotated by natural position (the oracle's rotation, rounded to
    the inputs' dtype as the in-place rotation stores it) and dq, dk are rotated back."""
    import oracle

    q, k = x["q"], x["k"]
    if rope_base:
        q = torch.from_numpy(oracle.rope(q, n, layout, rope_base)).to(x["q"].dtype)
        k = torch.from_numpy(oracle.rope(k, n, layout, rope_base)).to(x["k"].dtype)
    o, l = oracle.attn_fwd(q, k, x["v"], n, causal, layout)
    dq, dk, dv = oracle.attn_bwd(q, k, x["v"], x["dout"], n, causal, layout)
    if rope_base:
        dq = oracle.rope(dq, n, layout, rope_base, inverse=True)
        dk = oracle.rope(dk, n, layout, rope_base, inverse=True)
    return o, l, dq, dk, dv


def run_rank(rank, world, port, cases, device, result_dir, groups=None):
    """One rank: every case is (B, H, Hkv, L, d, causal, layout, dtype name, grad dtype name, seed[,
    rope base]); with a rope base the rank rotates its q and k shards before the ring and its dq, dk
    back after it (GPU ranks only).  With `groups`, the hierarchical ring (ring_fwd_2d / ring_bwd_2d
    over that many groups) instead of the flat one."""
    os.environ.setdefault("GLOO_SOCKET_IFNAME", "lo")
    ok = True
    try:
        dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
        import oracle
        from sequence_sharded_exact_gb300 import ring, synth

        if device != "cpu":
            torch.cuda.set_device(0)
        comm = ring.RingComm()
        assert comm.rank == rank and comm.world == world and comm.next == (rank + 1) % world
        n = world
        grid = ring.RingGrid(comm, groups) if groups else None

        def fwd(q_, k_, v_, causal_, layout_, **kw):
            if grid is None:
                return ring.ring_fwd(q_, k_, v_, comm, causal_, layout_, **kw)
            return ring.ring_fwd_2d(q_, k_, v_, grid, causal_, layout_, **kw)

        def bwd(q_, k_, v_, o_, l_, do_, causal_, layout_, **kw):
            if grid is None:
                return ring.ring_bwd(q_, k_, v_, o_, l_, do_, comm, causal_, layout_, **kw)
            return ring.ring_bwd_2d(q_, k_, v_, o_, l_, do_, grid, causal_, layout_, **kw)

        # the block each step computes: (rank - r) mod n on the flat ring, grid.held(a, b) on the grid
        order = ([(rank - r) % n for r in range(n)] if grid is None else
                 [grid.held(a, b) for a in range(grid.P) for b in range(grid.Q)])
        for case in cases:
            (B, H, Hkv, L, d, causal, layout, dt, gdt, seed), rope_base = case[:10], (case[10:] or (0.0,))[0]
            dtype = getattr(torch, dt)
            gdtype = getattr(torch, gdt)
            x = synth.make_inputs(B, H, Hkv, L, d, dtype=dtype, seed=seed, with_dout=True)
            ref_file = os.path.join(result_dir, f"ref_{seed}.npz")
            if os.path.exists(ref_file):  # precomputed once by the launching process
                z = np.load(ref_file)
                ref_o, ref_l, rq, rk, rv = (z[t] for t in ("o", "l", "dq", "dk", "dv"))
            else:
                ref_o, ref_l, rq, rk, rv = reference(x, n, causal, layout, rope_base)
            S = L // n
            sl = slice(rank * S, (rank + 1) * S)
            mine = {t: shard(x[t], rank, n) for t in ("q", "k", "v", "dout")}
            if device == "cpu":
                ops = OracleOps(L)
                out, lse = fwd(mine["q"], mine["k"], mine["v"], causal, layout, ops=ops)
                dq, dk, dv = bwd(mine["q"], mine["k"], mine["v"], out, lse, mine["dout"], causal, layout, ops=ops)
                # the schedule: the first block writes, later ones fold in; the backward stores each
                # contribution (the accumulators travel); every shard exactly once
                fcalls = [c for c in ops.calls if c[0] == "fwd"]
                bcalls = [c for c in ops.calls if c[0] == "bwd"]
                assert sorted(order) == list(range(n)), order
                assert fcalls == [("fwd", rank, j, r > 0) for r, j in enumerate(order)], fcalls
                assert bcalls == [("bwd", rank, j, False) for j in order], bcalls
                tol = {"out": 1e-10, "lse": 1e-10, "dq": 1e-10, "dk": 1e-10, "dv": 1e-10}
                rel = 1e-10
            else:
                from sequence_sharded_exact_gb300 import binding

                dev = torch.device("cuda", 0)
                g = {t: v.to(dev) for t, v in mine.items()}
                qr, kr = g["q"], g["k"]
                if rope_base:  # positions follow the blocks: each rank turns its own rows by natural position
                    qr = binding.block_rope(g["q"].clone(), n, rank, layout, base=rope_base)
                    kr = binding.block_rope(g["k"].clone(), n, rank, layout, base=rope_base)
                out, lse = fwd(qr, kr, g["v"], causal, layout)
                dq, dk, dv = bwd(qr, kr, g["v"], out, lse, g["dout"], causal, layout,
                                 grad_dtype=torch.float32 if rope_base else gdtype)
                if rope_base:  # gradients with respect to the unrotated q and k
                    binding.block_rope(dq, n, rank, layout, base=rope_base, inverse=True)
                    binding.block_rope(dk, n, rank, layout, base=rope_base, inverse=True)
                torch.cuda.synchronize()

                assert binding.device_status() == 0
                lim = 1e-4 if dtype == torch.float32 else 2e-2
                tol = {"out": lim, "lse": lim, "dq": lim, "dk": lim, "dv": lim}
                rel = 1.0 if dtype == torch.float32 else 5e-3
                if gdtype == torch.bfloat16:  # stored in bf16: its own rounding on top
                    for t in ("dq", "dk", "dv"):
                        tol[t] = None
            # the ring passes copies of the blocks on: the caller's own k and v are left as they were
            for t in ("k", "v"):
                held = mine[t] if device == "cpu" else g[t].cpu()
                assert torch.equal(held, shard(x[t], rank, n)), f"the ring overwrote the caller's {t}"
            got = {"out": out, "lse": lse, "dq": dq, "dk": dk, "dv": dv}
            ref = {"out": ref_o[:, :, sl], "lse": ref_l[:, :, sl], "dq": rq[:, :, sl], "dk": rk[:, :, sl],
                   "dv": rv[:, :, sl]}
            for name in got:
                gv = got[name].detach().double().cpu().numpy()
                ma, rl = errors(gv, ref[name])
                if tol[name] is None:
                    excess = np.abs(gv - ref[name]) - (2e-2 + np.abs(ref[name]) * 2.0 ** -8)
                    assert excess.max() <= 0 and rl <= 5e-3, f"{name}: {excess.max():.3e} {rl:.3e}"
                else:
                    assert ma <= tol[name] and rl <= rel, \
                        f"rank {rank}/{world} {layout} causal={causal} {dt} {name}: max-abs {ma:.3e}, rel-L2 {rl:.3e}"
        dist.barrier()
    except Exception:
        ok = False
        with open(os.path.join(result_dir, f"rank{rank}.err"), "w") as f:
            f.write(traceback.format_exc())
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()
    if ok:
        open(os.path.join(result_dir, f"rank{rank}.ok"), "w").close()


def precompute_refs(world, cases, result_dir):
    """The oracle of every case's whole sequence, computed once here for all ranks."""
    import oracle
    from sequence_sharded_exact_gb300 import synth

    for case in cases:
        (B, H, Hkv, L, d, causal, layout, dt, gdt, seed), rope_base = case[:10], (case[10:] or (0.0,))[0]
        x = synth.make_inputs(B, H, Hkv, L, d, dtype=getattr(torch, dt), seed=seed, with_dout=True)
        o, l, dq, dk, dv = reference(x, world, causal, layout, rope_base)
        np.savez(os.path.join(result_dir, f"ref_{seed}.npz"), o=o, l=l, dq=dq, dk=dk, dv=dv)


def launch(world, cases, device, result_dir, timeout=600, groups=None):
    """Spawns `world` ranks running run_rank and returns (all ok, error texts)."""
    import torch.multiprocessing as mp

    port = free_port()
    ctx = mp.start_processes(run_rank, args=(world, port, cases, device, result_dir, groups), nprocs=world,
                             join=False, start_method="spawn")
    import time

    t0 = time.time()
    while not ctx.join(timeout=5):
        if time.time() - t0 > timeout:
            for p in ctx.processes:
                if p.is_alive():
                    p.kill()
            return False, ["timed out"]
    errs = []
    for r in range(world):
        e = os.path.join(result_dir, f"rank{r}.err")
        if os.path.exists(e):
            errs.append(open(e).read())
    oks = all(os.path.exists(os.path.join(result_dir, f"rank{r}.ok")) for r in range(world))
    return oks and not errs, errs


def run_failing_rank(rank, world, port, mode, result_dir):
    """Failure detection on the ring (host side, gloo, no GPU): rank 1 leaves before its first transfer
    ("exit") or stops answering ("stall"); the other ranks' ring_fwd must end with an error within the
    process group's timeout instead of waiting for ever.  Writes rank<r>.detected with the seconds it
    took, or rank<r>.err."""
    import datetime
    import time

    os.environ.setdefault("GLOO_SOCKET_IFNAME", "lo")
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=5))
    from sequence_sharded_exact_gb300 import ring, synth

    comm = ring.RingComm()
    L = 48
    x = synth.make_inputs(1, 2, 1, L, 8, dtype=torch.float32, seed=3)
    mine = {t: shard(x[t], rank, world) for t in ("q", "k", "v")}
    if rank == 1:
        if mode == "exit":
            os._exit(0)  # leaves between steps: nothing of it is in flight
        time.sleep(3600)  # stalls; the launcher kills it
    t0 = time.time()
    try:
        ring.ring_fwd(mine["q"], mine["k"], mine["v"], comm, True, "zigzag", ops=OracleOps(L))
        with open(os.path.join(result_dir, f"rank{rank}.err"), "w") as f:
            f.write("ring_fwd returned although a neighbour was gone")
    except Exception as e:  # the transfer failed: the failure was detected
        with open(os.path.join(result_dir, f"rank{rank}.detected"), "w") as f:
            f.write(f"{time.time() - t0:.2f} {type(e).__name__}: {str(e)[:200]}")
    os._exit(0)  # no orderly shutdown: the group has lost a member


def run_autograd_rank(rank, world, port, groups, result_dir, device="cpu", causal=True, layout="zigzag",
                      module=False, f32_out=False):
    """ring_attention_distributed under autograd: the output and the gradients that backward() leaves
    on this rank's q, k, v equal its shard of the oracle's whole sequence.  CPU ranks use the oracle's
    block ops (float64, 1e-10); GPU ranks (sharing cuda:0) the library's kernels (bf16 inputs and
    gradients: the bf16 bounds, stored-bf16 for the gradients).  With ``module`` the call goes
    through the pages' per-rank object, RingAttention(dim, heads, rank, world_size); with ``f32_out``
    the forward's float32 running output is kept for the backward's D."""
    os.environ.setdefault("GLOO_SOCKET_IFNAME", "lo")
    try:
        dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
        import oracle
        from sequence_sharded_exact_gb300 import ring, synth

        comm = ring.RingComm()
        cpu = device == "cpu"
        B, H, Hkv, L, d = (1, 2, 1, 48, 8) if cpu else (1, 4, 2, 2048, 128)
        dt = torch.float32 if cpu else torch.bfloat16
        x = synth.make_inputs(B, H, Hkv, L, d, dtype=dt, seed=77, with_dout=True)
        ref_o, _ = oracle.attn_fwd(x["q"], x["k"], x["v"], world, causal, layout)
        rq, rk, rv = oracle.attn_bwd(x["q"], x["k"], x["v"], x["dout"], world, causal, layout)
        S = L // world
        sl = slice(rank * S, (rank + 1) * S)
        if cpu:
            q, k, v = (shard(x[t], rank, world).double().requires_grad_(True) for t in ("q", "k", "v"))
            do, ops = shard(x["dout"], rank, world).double(), OracleOps(L)
        else:
            torch.cuda.set_device(0)
            q, k, v = (shard(x[t], rank, world).cuda().requires_grad_(True) for t in ("q", "k", "v"))
            do, ops = shard(x["dout"], rank, world).cuda(), None
        if module:
            att = ring.RingAttention(H * d, H, rank, world, causal=causal, layout=layout, groups=groups, ops=ops,
                                     f32_out=f32_out)
            out = att(q, k, v)
            for bad in (dict(rank=(rank + 1) % world, world_size=world), dict(rank=rank, world_size=world + 1)):
                try:
                    ring.RingAttention(H * d, H, **bad)
                    raise AssertionError(f"RingAttention accepted {bad}")
                except ValueError:
                    pass
            try:
                ring.RingAttention(H * d // 2, H, rank, world)(q, k, v)   # head dim half of q's
                raise AssertionError("RingAttention accepted q with the wrong head dim")
            except ValueError:
                pass
        else:
            out = ring.ring_attention_distributed(q, k, v, comm, causal, layout, groups=groups, ops=ops,
                                                  f32_out=f32_out)
        (out.float() * do.float()).sum().backward()
        for got, ref, name in ((out.detach(), ref_o[:, :, sl], "out"), (q.grad, rq[:, :, sl], "dq"),
                               (k.grad, rk[:, :, sl], "dk"), (v.grad, rv[:, :, sl], "dv")):
            g = got.double().cpu().numpy()
            if cpu:
                err = float(np.abs(g - ref).max())
                assert err < 1e-10, f"rank {rank} {name}: {err:.3e}"
            else:
                assert got.dtype == torch.bfloat16
                excess = float((np.abs(g - ref) - (2e-2 + np.abs(ref) * 2.0 ** -8)).max())
                ma, rl = errors(g, ref)
                assert excess <= 0 and rl <= 5e-3, f"rank {rank} {name}: max-abs {ma:.3e}, rel-L2 {rl:.3e}"
        dist.barrier()
        open(os.path.join(result_dir, f"rank{rank}.ok"), "w").close()
    except Exception:
        with open(os.path.join(result_dir, f"rank{rank}.err"), "w") as f:
            f.write(traceback.format_exc())
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()
