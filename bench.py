"""Benchmark of the Ring Attention hot path on GB300 (prints ONE JSON line on rank 0).

Default workload: the long-context forward -- B=1, H=32 query heads, Hkv=8, d=128, L=131072 cut
into n=8 shards of 16384, causal, zigzag layout, bf16, 1% of key rows x8 -- i.e. the
configuration the throughput target is stated on.  One step = one ring-attention forward over the
whole sequence (one launch of the fused tensor-core kernel).  Secondary measurements in the same
line: the training workload (L=65536, n=16, forward + backward), the step-by-step ring (ring-step
kernel + LSE merge per step) on the long-context workload, and the merge kernel's bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {gb300,reference}] [--no-extra]

--impl reference times the float64 CPU oracle on a bounded sample of the same workload.
For N > 1 (torchrun, one rank per GPU) the workload is split over the N devices as the pages
describe: n = N shards of L / N tokens, one per device, each device computing its shard's block
attention against the K/V block it holds and passing the block round the ring over NCCL while it
computes (sequence_sharded_exact_gb300.ring); value = the whole sequence's work / the slowest
rank's time (strong scaling: the same workload at every N).  --ring runs that path at N = 1 too (one
device, one block); --replicas gives the older mode, one independent copy of the workload per rank.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "zigzag_gqa_128k"
TRAIN_WORKLOAD = "zigzag_gqa_64k_train"
METRIC = "ring-attention fwd/bwd TFLOP/s at 1 GB300 and % of dense BF16 tensor peak"

# DRAM bytes (read + write) per launch of the dominant kernel, measured by ncu on one launch at the
# bench size (summaries in profiles/: fwd_tc_kernel_zigzag_gqa_128k_metrics.md,
# bwd_tc_kernel_zigzag_gqa_64k_train_metrics.md, bwd_tc_kernel_striped_gqa_64k_train_metrics.md; the
# mean of the captures listed there).  Update or drop an entry whenever that kernel changes; a
# workload without an entry reports null.
TRAFFIC_BYTES = {("zigzag_gqa_128k", "fwd"): 3.765638144e9 + 1.081261056e9,
                 ("zigzag_gqa_64k_train", "train"): 7.372813995e9 + 3.979190101e9,
                 ("striped_gqa_64k_train", "train"): 6.576252672e9 + 3.563336192e9}


def copy_bandwidth(host, device_t, stream):
    """This box's pinned host <-> device copy rates (GB/s), one large copy each way on `stream`: the
    end-to-end number depends on them (machines in the same pool have differed by 10x)."""
    n = min(host.numel(), device_t.numel())
    h, d = host.view(-1)[:n], device_t.view(-1)[:n]
    nbytes = n * host.element_size()
    rates = {}
    for name, (dst, src) in (("h2d", (d, h)), ("d2h", (h, d))):
        with torch.cuda.stream(stream):
            dst.copy_(src, non_blocking=True)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dst.copy_(src, non_blocking=True)
            b.record(stream)
        b.synchronize()
        rates[name] = round(nbytes / (a.elapsed_time(b) / 1e3) / 1e9, 1)
    return rates


def fwd_flops(B, H, L, d, causal):
    """Algorithmic forward flops: 4 B H L^2 d (QK^T and PV), halved when causal."""
    f = 4.0 * B * H * L * L * d
    return f / 2 if causal else f


def max_over_ranks(value, dist_mod=None, device="cpu"):
    """The largest of every rank's value (identity without a process group)."""
    if dist_mod is None:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
    return float(t.item())


def visible_tile_flops(B, H, L, d, n, causal, layout, tile=128):
    """Forward flops of every (query tile, key tile) pair with at least one visible (q, k) element at
    the kernels' 128-row tiles, each counted whole (diagonal tiles in full): what the tensor cores
    execute at the least.  The algorithmic count (fwd_flops) halves the diagonal tiles instead."""
    import sequence_sharded_exact_gb300 as ra

    tiles = sum(ra.shard_tiles(L, n, causal, layout, tile))
    return 4.0 * B * H * tiles * tile * tile * d


def whole_job_tflops(world, flops_per_step, steps, max_total_ms):
    """All ranks' algorithmic work over the slowest rank's time, in TFLOP/s."""
    return world * flops_per_step * steps / (max_total_ms / 1e3) / 1e12


# NVIDIA's published dense BF16 tensor-core rate of one GB300 (Blackwell Ultra) GPU: the GB300 NVL72
# figure of 360 PFLOPS FP16/BF16 for 72 GPUs is quoted with 2:4 sparsity, i.e. 2.5 PFLOP/s dense per
# GPU (the HGX B300 figure of 36 PFLOPS for 8 GPUs, also sparse, gives 2.25 dense per GPU).
PUBLISHED_BF16_DENSE_TFLOPS = 2500.0
PUBLISHED_BF16_SOURCE = ("NVIDIA GB300 NVL72 specifications: 360 PFLOPS FP16/BF16 tensor (with sparsity) for "
                         "72 GPUs = 2.5 PFLOP/s dense per GPU")
# Dense bf16 tcgen05 rate per SM and clock: one 128 x 128 x 16 MMA (524288 flop) every 64 cycles,
# measured on this GPU with a microbenchmark of back-to-back tcgen05.mma instructions.
FLOP_PER_CLK_PER_SM = 8192


def per_clock_peak_tflops(sm_mhz):
    """SMs x 8192 flop/clock x the SM clock sampled under load (TFLOP/s), or None."""
    if not sm_mhz or not torch.cuda.is_available():
        return None
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return sms * FLOP_PER_CLK_PER_SM * sm_mhz * 1e6 / 1e12


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p["bf16_tflops"], p["bf16_tflops_sustained"], p["hbm_gbs"], "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def time_launches(fn, steps, warmup, stream):
    """Warm up, then time `steps` calls with CUDA events on `stream`; returns per-call ms list."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def sample_rows(B, H, L, count, seed):
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(B * H * L, size=count, replace=False))


def oracle_calibrate(x, w, target_s, seed=7):
    """Number of random query rows the float64 oracle handles in about target_s seconds."""
    import oracle

    B, H, L, n = w["B"], w["H"], w["L"], w["n"]
    arrs = tuple(x[t].float().cpu().numpy() for t in ("q", "k", "v"))
    count, limit = 32, B * H * L // 4
    while True:
        rows = sample_rows(B, H, L, count, seed)
        t0 = time.perf_counter()
        oracle.attn_fwd_rows(*arrs, n, w["causal"], w["layout"], rows)
        dt = time.perf_counter() - t0
        if dt >= target_s / 8 or count >= limit:
            break
        count = int(min(limit, count * 2))
    return arrs, max(16, min(limit, int(count * target_s / max(dt, 1e-3))))


def oracle_sample(arrs, w, count, seed):
    """Times the float64 oracle on `count` random query rows of the workload.
    Returns (TFLOP/s, seconds, rows, cores, algorithmic flops of those rows)."""
    import oracle

    B, H, L, d, n = w["B"], w["H"], w["L"], w["d"], w["n"]
    rows = sample_rows(B, H, L, count, seed)
    t0 = time.perf_counter()
    oracle.attn_fwd_rows(*arrs, n, w["causal"], w["layout"], rows)
    dt = time.perf_counter() - t0
    flops = sum(row_flops(int(r), B, H, L, d, n, w["causal"], w["layout"]) for r in rows)
    return flops / dt / 1e12, dt, len(rows), oracle.num_threads(), flops


def row_flops(idx, B, H, L, d, n, causal, layout):
    """Algorithmic flops of one query row: 4 d per visible key."""
    import oracle

    if not causal:
        return 4.0 * d * L
    p = oracle.natural_position(idx % L, L, n, layout)
    return 4.0 * d * (p + 1)


def run_reference(args, w):
    """--impl reference: the float64 CPU oracle, timed on bounded samples of the workload."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    ring_mode = args.ring or (world > 1 and not args.replicas)
    if ring_mode:
        w = dict(w, n=world)  # the same sequence cut into one shard per rank, as the ring arm runs it
    from sequence_sharded_exact_gb300 import synth

    gen = "cuda" if torch.cuda.is_available() else "cpu"
    x = synth.make_inputs(w["B"], w["H"], w["Hkv"], w["L"], w["d"], dtype=w["dtype"],
                          seed=w["seed"], spike_frac=w["spike_frac"], device="cpu", gen_device=gen)
    per_step = max(2.0, 90.0 / max(1, args.steps + args.warmup))
    arrs, count = oracle_calibrate(x, w, per_step)
    del x
    secs, rows_total, cores, flops_total = 0.0, 0, 1, 0.0
    for s in range(args.warmup + args.steps):
        _, dt, rows, cores, flops = oracle_sample(arrs, w, count, seed=100 + s)
        if s >= args.warmup:
            secs += dt
            rows_total += rows
            flops_total += flops
    value = flops_total / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / max(1, args.steps) * 1e3, "higher_is_better": True,
        "scaling": "strong" if ring_mode else "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": ring_config(w, world, args) if ring_mode else config_dict(w, args.step),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{count} random query rows of the workload per step, "
                                   f"{args.steps} timed steps (float64 two-pass attention rows)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict(w, step="fwd"):
    return {"workload": f"ring attention {'fwd+bwd' if step == 'train' else 'fwd'}, B{w['B']} H{w['H']} Hkv{w['Hkv']} d{w['d']} "
                        f"L{w['L']} n{w['n']} {'causal' if w['causal'] else 'full'} {w['layout']}",
            "B": w["B"], "H": w["H"], "Hkv": w["Hkv"], "L": w["L"], "d": w["d"], "n_shards": w["n"],
            "causal": w["causal"], "layout": w["layout"], "tile": 128,
            "key_rows_x8": w["spike_frac"], "seed": w["seed"],
            "l2": f"inputs ({(w['H'] + 2 * w['Hkv']) * w['B'] * w['L'] * w['d'] * 2 / 1e9:.2f} GB) "
                  "larger than L2; no flush"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary measurements")
    ap.add_argument("--oracle-seconds", type=float, default=15.0)
    ap.add_argument("--workload", default=None,
                    help="synthetic workload name (default: the long-context forward for --step "
                         "fwd, the 64K training workload for --step train)")
    ap.add_argument("--seed", type=int, default=None,
                    help="seed of the synthetic inputs (default: the workload's own)")
    ap.add_argument("--step", default="fwd", choices=["fwd", "train"],
                    help="fwd: one ring-attention forward per step; train: forward + backward")
    ap.add_argument("--ring", action="store_true",
                    help="run the multi-device ring path also at N = 1 (the default for N > 1)")
    ap.add_argument("--replicas", action="store_true",
                    help="N > 1: one independent copy of the workload per rank instead of the ring")
    ap.add_argument("--dist-backend", default="nccl", choices=["nccl", "gloo"],
                    help="N > 1 ring: the process group's backend (gloo stages the blocks through host "
                         "memory; with fewer GPUs than ranks, ranks share devices round robin)")
    ap.add_argument("--ring-groups", type=int, default=1,
                    help="the ring as a hierarchical ring: a local ring inside each of this many groups "
                         "of consecutive ranks (e.g. the GPUs of one node), a global ring across them")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    from sequence_sharded_exact_gb300 import synth

    if args.workload is None:
        args.workload = WORKLOAD if args.step == "fwd" else TRAIN_WORKLOAD
    w = dict(synth.WORKLOADS[args.workload])
    if args.seed is not None:
        w["seed"] = args.seed
    if args.impl == "reference":
        run_reference(args, w)
        return

    import sequence_sharded_exact_gb300 as ra

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.ring or (world > 1 and not args.replicas):
        run_ring(args, w, world, rank, local)
        return
    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist = dist_mod
        torch.cuda.set_device(local)
        with _StdoutToStderr():
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream(dev)

    B, H, Hkv, L, d, n = w["B"], w["H"], w["Hkv"], w["L"], w["d"], w["n"]
    train = args.step == "train"
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=w["dtype"], seed=w["seed"] + rank,
                          spike_frac=w["spike_frac"], with_dout=train, device=dev, gen_device=dev)
    q, k, v = x["q"], x["k"], x["v"]
    out = torch.empty_like(q)
    lse = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    path = ra.fwd_path(B, H, Hkv, L, d, n, w["causal"], w["layout"], w["dtype"])
    ff = fwd_flops(B, H, L, d, w["causal"])
    flops = 3.5 * ff if train else ff
    dq = dk = dv = wsb = None
    if train:
        path += "+" + ra.bwd_path(B, H, Hkv, L, d, n, w["causal"], w["layout"], w["dtype"])
        dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
        dk = torch.empty(k.shape, dtype=torch.float32, device=dev)
        dv = torch.empty(v.shape, dtype=torch.float32, device=dev)
        wsb = torch.empty(max(256, ra.bwd_workspace_size(B, H, Hkv, L, d, torch.float32)),
                          dtype=torch.uint8, device=dev)

    def fwd_call():
        ra.fwd(q, k, v, n, w["causal"], w["layout"], out=out, lse=lse, stream=stream)

    def bwd_call():
        ra.bwd(q, k, v, out, lse, x["dout"], n, w["causal"], w["layout"], dq=dq, dk=dk, dv=dv,
               workspace=wsb, stream=stream)

    def step():
        fwd_call()
        if train:
            bwd_call()

    # timed region: barrier + synchronize on both sides, CUDA events on the launch stream
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        per = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(args.steps)]
        ev0.record(stream)
        for a, b, c in per:
            a.record(stream)
            fwd_call()
            b.record(stream)
            if train:
                bwd_call()
            c.record(stream)
        ev1.record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    total_ms = ev0.elapsed_time(ev1)
    fwd_ms = [a.elapsed_time(b) for a, b, _ in per]
    bwd_ms = [b.elapsed_time(c) for _, b, c in per] if train else []
    status = ra.device_status()
    total_ms = max_over_ranks(total_ms, dist, dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_tflops(world, flops, args.steps, total_ms)

    peak_b, peak_s, hbm, peak_kind = peaks()
    if train:
        kname, kflops, kms = "bwd_tc_kernel", 2.5 * ff, statistics.mean(bwd_ms)
        note = "ring_attn_bwd call (preprocess + zero + bwd_tc_kernel), CUDA events"
    else:
        kname, kflops, kms = "fwd_tc_kernel", ff, statistics.mean(fwd_ms)
        note = "one fwd_tc_kernel launch, CUDA events"
    achieved = kflops / (kms / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: q,k,v ~ N(0,1) bf16" + (", 1% of key rows x8" if w["spike_frac"] else "")
                + (", dO ~ N(0,1)" if train else "") + ", seeded",
        "config": config_dict(w, args.step),
        "fraction_of_peak": value / world / peak_b,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_b, "unit": "TFLOP/s",
                     "frac": achieved / peak_b,
                     "traffic": TRAFFIC_BYTES.get((args.workload, args.step)),
                     "peak_kind": f"{peak_kind} bf16 burst (MEASURED_PEAKS bf16_tflops)",
                     "frac_of_sustained": achieved / peak_s,
                     "kernel": kname, "timed": note, "algorithmic_flops_per_launch": kflops,
                     "visible_tile_flops_per_launch": (2.5 if train else 1.0) * visible_tile_flops(
                         B, H, L, d, n, w["causal"], w["layout"])},
        "gpu_launches": args.steps * (4 if train else 1),
        "path": path,
        "device_status": status,
    }
    if train:
        line["fwd_ms"] = statistics.mean(fwd_ms)
        line["bwd_ms"] = statistics.mean(bwd_ms)

    # end to end: pinned host buffers -> device, the C-ABI calls, results -> host, every step
    if rank == 0 or dist:
        ins = [q, k, v] + ([x["dout"]] if train else [])
        outs = [dq, dk, dv] if train else [out, lse]
        h_in = [t.cpu().pin_memory() for t in ins]
        h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]

        if train:
            def e2e_step():
                for dst, src in zip(ins, h_in):
                    dst.copy_(src, non_blocking=True)
                step()
                for dst, src in zip(h_out, outs):
                    dst.copy_(src, non_blocking=True)
            what = "forward + backward through the C ABI with pinned host buffers in and out"
        else:
            # ring_attn_fwd_host: host buffers in and out, the copies of one kv-head group overlapped
            # with the compute of the others
            hws = torch.empty(ra.library().ring_attn_fwd_host_workspace_size(H, Hkv, L, d, 1),
                              dtype=torch.uint8, device=dev)

            def e2e_step():
                ra.fwd_host(h_in[0], h_in[1], h_in[2], n, w["causal"], w["layout"], out=h_out[0], lse=h_out[1],
                            workspace=hws, device=dev, stream=stream)
            what = ("forward through ring_attn_fwd_host: pinned host buffers in and out, copies overlapped "
                    "with the compute of other kv-head groups")

        e2e_steps = max(2, args.steps // 2)
        with ClockSampler(dev.index) as e2e_clk:
            e2e_ms = sum(time_launches(e2e_step, e2e_steps, 1, stream)) / e2e_steps
        h2d = sum(t.numel() * t.element_size() for t in h_in)
        d2h = sum(t.numel() * t.element_size() for t in h_out)
        line["e2e"] = {"value": world * flops / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s", "what": what,
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "ms_per_step": e2e_ms, "copy_GBps": copy_bandwidth(h_in[0], ins[0], stream),
                       "clocks": e2e_clk.summary()}
        if not train:
            # the results that came back match the device-resident forward of the timed region
            line["e2e"]["matches_device_forward"] = bool(torch.equal(h_out[0], out.cpu()) and
                                                         torch.equal(h_out[1], lse.cpu()))
            del hws
        del h_in, h_out

    line["clocks"] = clk.summary()
    add_peak_fractions(line["roofline"], line["clocks"])

    if rank == 0 and not args.no_extra and not train:
        line["extra"] = secondary(ra, w, x, out, lse, stream, dev, peak_b, hbm, args)
    if rank == 0 and world == 1:
        arrs, count = oracle_calibrate(x, w, args.oracle_seconds)
        tf, secs, rows, cores, oflops = oracle_sample(arrs, w, count, seed=11)
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                                "sample": f"{rows} random query rows of the workload "
                                          f"({oflops / 1e9:.1f} GFLOP, {secs:.1f} s, float64)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def add_peak_fractions(roof, clocks):
    """The roofline's other denominators: the per-clock tensor peak at the SM clock sampled under load
    (SMs x 8192 flop/clock x MHz: it separates what the kernel does per cycle from the clock the power
    cap allows) and NVIDIA's published dense BF16 figure."""
    pc = per_clock_peak_tflops(clocks.get("sm_mhz"))
    roof["per_clock_peak"] = pc
    roof["frac_of_per_clock_peak"] = roof["achieved"] / pc if pc else None
    roof["per_clock_peak_how"] = f"SMs x {FLOP_PER_CLK_PER_SM} flop/clock x median sampled SM MHz"
    roof["published_peak"] = PUBLISHED_BF16_DENSE_TFLOPS
    roof["frac_of_published_peak"] = roof["achieved"] / PUBLISHED_BF16_DENSE_TFLOPS
    roof["published_peak_source"] = PUBLISHED_BF16_SOURCE


class TimedOps:
    """The ring's library calls with CUDA events around every block forward / backward launch, so that
    the dominant kernel's own launch time can be reported."""

    def __init__(self, stream):
        from sequence_sharded_exact_gb300 import ring

        self.inner = ring.LibraryOps(stream)
        self.stream = stream
        self.events = {"fwd": [], "bwd": []}
        self.record = False

    def __getattr__(self, name):
        return getattr(self.inner, name)

    def _timed(self, kind, fn, *a):
        if not self.record:
            return fn(*a)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        fn(*a)
        e1.record(self.stream)
        self.events[kind].append((e0, e1))

    def block_fwd(self, *a):
        self._timed("fwd", self.inner.block_fwd, *a)

    def block_bwd(self, *a):
        self._timed("bwd", self.inner.block_bwd, *a)

    def mean_ms(self, kind):
        ev = self.events[kind]
        return statistics.mean(a.elapsed_time(b) for a, b in ev) if ev else None


class _StdoutToStderr:
    """Routes file descriptor 1 to 2 while open: the process-group setup of some backends prints
    status lines on stdout, where the bench prints only its JSON line."""

    def __enter__(self):
        sys.stdout.flush()
        self.saved = os.dup(1)
        os.dup2(2, 1)
        return self

    def __exit__(self, *exc):
        sys.stdout.flush()
        os.dup2(self.saved, 1)
        os.close(self.saved)
        return False


def ring_config(w, world, args):
    """The config of the ring mode: the workload cut into one shard per rank (the reference arm
    reports the same)."""
    B, H, Hkv, L, d = w["B"], w["H"], w["Hkv"], w["L"], w["d"]
    S = L // world
    shard_bytes = (H + 2 * Hkv) * B * S * d * 2
    ngpu = torch.cuda.device_count()
    return dict(config_dict(dict(w, n=world), args.step),
                parallelism=f"context parallel: ring over {world} device(s), one shard of {S} tokens each"
                            + (f", hierarchical: {args.ring_groups} groups of {world // args.ring_groups}"
                               if args.ring_groups > 1 else ""),
                l2=f"each rank's shard of q, k, v ({shard_bytes / 1e9:.2f} GB) "
                   + ("larger than L2; no flush" if shard_bytes > 129e6
                      else "smaller than L2 (129 MB): repeated steps may hit in L2"),
                mode=(f"multi-device ring (blocks over {args.dist_backend.upper()}"
                      + (f", {world} ranks on {ngpu} GPU(s)" if world > ngpu else "") + ")")
                if world > 1 else "ring path on one device")


def run_ring(args, w, world, rank, local):
    """The multi-device ring: n = world shards of the workload's sequence, one per rank, blocks passed
    round the ring over NCCL (one rank per GPU; gloo only when torch has no NCCL)."""
    import torch.distributed as dist
    import sequence_sharded_exact_gb300 as ra
    from sequence_sharded_exact_gb300 import ring, synth

    torch.cuda.set_device(local % torch.cuda.device_count() if world > 1 else 0)
    dev = torch.device("cuda", torch.cuda.current_device())
    with _StdoutToStderr():
        if world > 1 and args.dist_backend == "nccl":
            dist.init_process_group("nccl", device_id=dev)
        elif world > 1:
            dist.init_process_group("gloo")
        else:
            dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % free_port(), rank=0, world_size=1)
    comm = ring.RingComm()
    grid = ring.RingGrid(comm, args.ring_groups) if args.ring_groups > 1 else None
    rfwd = (lambda *a, **kw: ring.ring_fwd(*a[:3], comm, *a[3:], **kw)) if grid is None else \
        (lambda *a, **kw: ring.ring_fwd_2d(*a[:3], grid, *a[3:], **kw))
    rbwd = (lambda *a, **kw: ring.ring_bwd(*a[:6], comm, *a[6:], **kw)) if grid is None else \
        (lambda *a, **kw: ring.ring_bwd_2d(*a[:6], grid, *a[6:], **kw))
    stream = torch.cuda.current_stream(dev)
    B, H, Hkv, L, d = w["B"], w["H"], w["Hkv"], w["L"], w["d"]
    n, causal, layout = world, w["causal"], w["layout"]
    if layout == "zigzag" and L % (2 * n):
        raise SystemExit(f"L = {L} does not split into 2 x {n} zigzag chunks")
    train = args.step == "train"
    # every rank draws the same whole-sequence inputs (seeded) and keeps its own shard's rows
    x = synth.make_inputs(B, H, Hkv, L, d, dtype=w["dtype"], seed=w["seed"], spike_frac=w["spike_frac"],
                          with_dout=train, device=dev, gen_device=dev)
    S = L // n
    mine = {t: x[t][:, :, rank * S:(rank + 1) * S].contiguous() for t in x}
    del x
    torch.cuda.empty_cache()
    ops = TimedOps(stream)
    ff = fwd_flops(B, H, L, d, causal)
    flops = 3.5 * ff if train else ff
    res = {}

    def step():
        out, lse = rfwd(mine["q"], mine["k"], mine["v"], causal, layout, ops=ops)
        if train:
            rbwd(mine["q"], mine["k"], mine["v"], out, lse, mine["dout"], causal, layout, ops=ops)
        res["out"], res["lse"] = out, lse

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    ops.record = True
    with ClockSampler(dev.index) as clk:
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
    ops.record = False
    dist.barrier()
    torch.cuda.synchronize()
    total_ms = max_over_ranks(ev0.elapsed_time(ev1), dist if world > 1 else None, dev)
    status = ra.device_status()
    value = flops * args.steps / (total_ms / 1e3) / 1e12  # the whole sequence's work, all ranks together
    peak_b, peak_s, hbm, peak_kind = peaks()
    kind = "bwd" if train else "fwd"
    kms = ops.mean_ms(kind)
    per_launch = (2.5 * ff if train else ff) / (n * n)  # each rank runs n of the n^2 blocks per pass
    achieved = per_launch / (kms / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: q,k,v ~ N(0,1) bf16" + (", 1% of key rows x8" if w["spike_frac"] else "")
                + (", dO ~ N(0,1)" if train else "") + ", seeded",
        "config": ring_config(w, world, args),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_b, "unit": "TFLOP/s",
                     "frac": achieved / peak_b, "traffic": None,
                     "peak_kind": f"{peak_kind} bf16 burst (MEASURED_PEAKS bf16_tflops)",
                     "kernel": "bwd_tc_kernel (block calls)" if train else "fwd_tc_kernel (block calls)",
                     "timed": f"mean of the {kind} block launches of rank {rank}, CUDA events",
                     "algorithmic_flops_per_launch": per_launch},
        # forward: n block launches + 1 conversion; backward: preprocess, zero, n blocks, 2 (n - 1) adds
        # of the travelling dK / dV accumulators, 3 conversions
        "gpu_launches": args.steps * (n + 1 + (3 * n + 3 if train else 0)),
        "device_status": status,
    }
    line["clocks"] = clk.summary()
    add_peak_fractions(line["roofline"], line["clocks"])
    # end to end: this rank's shard from pinned host memory, the ring, its results back to the host
    h_in = {t: mine[t].cpu().pin_memory() for t in mine}
    h_out = [torch.empty(res["out"].shape, dtype=res["out"].dtype, pin_memory=True),
             torch.empty(res["lse"].shape, dtype=torch.float32, pin_memory=True)]
    d_in = {t: torch.empty_like(mine[t]) for t in mine}

    def e2e_step():
        for t in mine:
            d_in[t].copy_(h_in[t], non_blocking=True)
        out, lse = rfwd(d_in["q"], d_in["k"], d_in["v"], causal, layout, ops=ops)
        if train:
            rbwd(d_in["q"], d_in["k"], d_in["v"], out, lse, d_in["dout"], causal, layout, ops=ops)
        h_out[0].copy_(out, non_blocking=True)
        h_out[1].copy_(lse, non_blocking=True)

    e2e_steps = max(2, args.steps // 2)
    for _ in range(1):
        e2e_step()
    torch.cuda.synchronize()
    dist.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    t1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(t0.elapsed_time(t1), dist if world > 1 else None, dev) / e2e_steps
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    line["e2e"] = {"value": flops / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                   "what": "every rank: its shard from pinned host memory, the ring, its out and lse back",
                   "h2d_bytes_per_step": h2d * world, "d2h_bytes_per_step": d2h * world, "ms_per_step": e2e_ms}
    if rank == 0:
        print(json.dumps(line), flush=True)
    dist.barrier()
    dist.destroy_process_group()


def free_port():
    import socket

    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def other_workload(ra, name, stream, dev, peak_b):
    """Forward (and, for a training workload, forward + backward) of another synthetic workload:
    TFLOP/s and the fraction of the measured bf16 peak, 3 timed calls after 1 warm-up."""
    from sequence_sharded_exact_gb300 import synth

    ww = synth.WORKLOADS[name]
    B, H, Hkv, L, d, n = ww["B"], ww["H"], ww["Hkv"], ww["L"], ww["d"], ww["n"]
    xx = synth.make_workload(name, device=dev, gen_device=dev)
    o, l = ra.fwd(xx["q"], xx["k"], xx["v"], n, ww["causal"], ww["layout"])
    ff = fwd_flops(B, H, L, d, ww["causal"])
    fms = statistics.mean(time_launches(lambda: ra.fwd(xx["q"], xx["k"], xx["v"], n, ww["causal"], ww["layout"],
                                                       out=o, lse=l, stream=stream), 3, 1, stream))
    res = {"workload": f"B{B} H{H} Hkv{Hkv} d{d} L{L} n{n} causal {ww['layout']}",
           "fwd_ms": fms, "fwd_tflops": ff / (fms / 1e3) / 1e12, "fwd_frac": ff / (fms / 1e3) / 1e12 / peak_b,
           "path": ra.fwd_path(B, H, Hkv, L, d, n, ww["causal"], ww["layout"], ww["dtype"])}
    if ww["backward"]:
        grads = [torch.empty(t.shape, dtype=torch.float32, device=dev) for t in (xx["q"], xx["k"], xx["v"])]
        wsb = torch.empty(max(256, ra.bwd_workspace_size(B, H, Hkv, L, d, torch.float32)), dtype=torch.uint8,
                          device=dev)
        bms = statistics.mean(time_launches(lambda: ra.bwd(xx["q"], xx["k"], xx["v"], o, l, xx["dout"], n, ww["causal"],
                                                           ww["layout"], dq=grads[0], dk=grads[1], dv=grads[2],
                                                           workspace=wsb, stream=stream), 3, 1, stream))
        res.update(bwd_ms=bms, bwd_tflops=2.5 * ff / (bms / 1e3) / 1e12, bwd_frac=2.5 * ff / (bms / 1e3) / 1e12 / peak_b,
                   train_tflops=3.5 * ff / ((fms + bms) / 1e3) / 1e12)
        del grads, wsb
    del xx, o, l
    return res


def secondary(ra, w, x, out, lse, stream, dev, peak_b, hbm, args):
    """Training workload (fwd + bwd), stepwise ring (steps folded into a running result), and the
    bandwidth of the HBM-bound kernels (LSE merge, backward preprocess, RoPE, Ulysses all-to-all)."""
    from sequence_sharded_exact_gb300 import synth

    res = {}
    B, H, Hkv, L, d, n = w["B"], w["H"], w["Hkv"], w["L"], w["d"], w["n"]
    steps = max(2, min(args.steps, 5))
    # stepwise ring: n ring-step launches (steps 1.. fold into the running result) + conversion
    ws = torch.empty(ra.library().ring_attn_fwd_stepwise_workspace_size(B, H, L, d),
                     dtype=torch.uint8, device=dev)
    out2, lse2 = torch.empty_like(out), torch.empty_like(lse)
    ms = time_launches(lambda: ra.fwd_stepwise(x["q"], x["k"], x["v"], n, w["causal"], w["layout"],
                                               out=out2, lse=lse2, workspace=ws, stream=stream),
                       steps, 1, stream)
    flops = fwd_flops(B, H, L, d, w["causal"])
    res["stepwise_fwd"] = {"tflops": flops / (statistics.mean(ms) / 1e3) / 1e12,
                           "ms": statistics.mean(ms), "launches": n + 1}
    # LSE merge kernel alone: bytes = rows * (3 d + 3) * 4 (read o_acc, o_part, write o_acc, lse)
    rows = B * H * L
    o_acc = ws[: rows * d * 4].view(torch.float32).view(rows, d)
    part = torch.randn(rows, d, device=dev)
    la = torch.randn(rows, device=dev)
    lb = torch.randn(rows, device=dev)
    ms = time_launches(lambda: ra.lse_merge(o_acc, la, part, lb, stream=stream), 10, 3, stream)
    gbytes = rows * (3 * d + 3) * 4 / 1e9
    res["lse_merge"] = {"GB/s": gbytes / (statistics.mean(ms) / 1e3), "peak_GB/s": hbm,
                        "frac": gbytes / (statistics.mean(ms) / 1e3) / hbm, "ms": statistics.mean(ms)}
    del ws, out2, lse2, part, la, lb, o_acc
    # backward preprocess D = rowsum(dO * O) alone, on the workload's out with q standing in for dO
    # (same shape and dtype); bytes = rows * (2 * d * 2 + 4) (read O and dO in bf16, write D)
    Dv = torch.empty((B, H, L), dtype=torch.float32, device=dev)
    ms = time_launches(lambda: ra.bwd_preprocess(out, x["q"], D=Dv, stream=stream), 10, 3, stream)
    gbytes = rows * (2 * d * out.element_size() + 4) / 1e9
    res["bwd_preprocess"] = {"GB/s": gbytes / (statistics.mean(ms) / 1e3), "peak_GB/s": hbm,
                             "frac": gbytes / (statistics.mean(ms) / 1e3) / hbm, "ms": statistics.mean(ms)}
    del Dv
    # rotary positions on a copy of the workload's q, in place; bytes = read + write of q per launch
    qr = x["q"].clone()
    qb = qr.numel() * qr.element_size()
    ms = time_launches(lambda: ra.rope(qr, n, w["layout"], stream=stream), 5, 2, stream)
    per = statistics.mean(ms)
    res["rope_q"] = {"GB/s": 2 * qb / 1e9 / (per / 1e3), "peak_GB/s": hbm,
                     "frac": 2 * qb / 1e9 / (per / 1e3) / hbm, "ms": per}
    del qr
    # Ulysses variant on the same workload: token split in, three all-to-alls, attention per shard
    # over the whole sequence, two all-to-alls back (Hkv must divide by n)
    if H % n == 0 and Hkv % n == 0 and w["d"] in (64, 128):
        S = L // n
        tok = lambda t: t.view(B, t.shape[1], n, S, d).permute(2, 0, 3, 1, 4).contiguous()
        qt, kt, vt = tok(x["q"]), tok(x["k"]), tok(x["v"])
        ot = torch.empty_like(qt)
        lt_ = torch.empty((n, B, S, H), dtype=torch.float32, device=dev)
        wsu = torch.empty(ra.library().ring_attn_ulysses_workspace_size(B, H, Hkv, L, d, 1), dtype=torch.uint8,
                          device=dev)
        ms = time_launches(lambda: ra.ulysses_fwd(qt, kt, vt, n, w["causal"], w["layout"], out=ot, lse=lt_,
                                                  workspace=wsu, stream=stream), 3, 1, stream)
        hs = torch.empty(n, B, H // n, L, d, dtype=qt.dtype, device=dev)
        ams = time_launches(lambda: ra.ulysses_a2a(qt, n, w["layout"], 0, dst=hs, stream=stream), 5, 2, stream)
        qbytes = qt.numel() * qt.element_size()
        res["ulysses_fwd"] = {"tflops": flops / (statistics.mean(ms) / 1e3) / 1e12, "ms": statistics.mean(ms),
                              "a2a_q_GB/s": 2 * qbytes / 1e9 / (statistics.mean(ams) / 1e3),
                              "a2a_q_ms": statistics.mean(ams)}
        del qt, kt, vt, ot, lt_, wsu, hs
    # causal work per shard: the host scheduler's tile counts for the contiguous 8K configuration and
    # for this workload, and the tile pairs the forward kernel computed on the device, per shard pair
    c8 = synth.WORKLOADS["causal_contig_8k"]
    sched = {}
    for name, ww in (("causal_contig_8k", c8), (args.workload, w)):
        for lay in ("contiguous", "zigzag", "striped"):
            if lay == "zigzag" and ww["L"] % (2 * ww["n"]):
                continue
            t = ra.shard_tiles(ww["L"], ww["n"], ww["causal"], lay)
            sched[f"{name}/{lay}"] = {"tiles_per_shard_per_head": t, "max_over_mean": max(t) / (sum(t) / len(t))}
    _, _, visits = ra.fwd_tile_visits(x["q"], x["k"], x["v"], n, w["causal"], w["layout"], stream=stream)
    per_shard = visits.sum(dim=1).tolist()
    sched["device_visits_" + w["layout"]] = {"tile_pairs_per_query_shard": per_shard,
                                             "max_over_mean": max(per_shard) / (sum(per_shard) / len(per_shard))}
    res["causal_work_per_shard"] = sched
    # training workload: forward + backward
    t = synth.WORKLOADS[TRAIN_WORKLOAD]
    xt = synth.make_workload(TRAIN_WORKLOAD, device=dev, gen_device=dev)
    Bt, Ht, Hkt, Lt, dt_, nt = t["B"], t["H"], t["Hkv"], t["L"], t["d"], t["n"]
    ot, lt = ra.fwd(xt["q"], xt["k"], xt["v"], nt, t["causal"], t["layout"])
    dq = torch.empty(xt["q"].shape, dtype=torch.float32, device=dev)
    dk = torch.empty(xt["k"].shape, dtype=torch.float32, device=dev)
    dv = torch.empty(xt["v"].shape, dtype=torch.float32, device=dev)
    wsb = torch.empty(max(256, ra.bwd_workspace_size(Bt, Ht, Hkt, Lt, dt_, torch.float32)),
                      dtype=torch.uint8, device=dev)

    def train_step():
        ra.fwd(xt["q"], xt["k"], xt["v"], nt, t["causal"], t["layout"], out=ot, lse=lt, stream=stream)
        ra.bwd(xt["q"], xt["k"], xt["v"], ot, lt, xt["dout"], nt, t["causal"], t["layout"],
               dq=dq, dk=dk, dv=dv, workspace=wsb, stream=stream)

    bwd_steps = 2 if ra.bwd_path(Bt, Ht, Hkt, Lt, dt_, nt, t["causal"], t["layout"],
                                 t["dtype"]) == "tcgen05" else 0
    ff = fwd_flops(Bt, Ht, Lt, dt_, t["causal"])
    if bwd_steps:
        ms = time_launches(train_step, bwd_steps, 1, stream)
        res["train_fwd_bwd"] = {"workload": f"B{Bt} H{Ht} Hkv{Hkt} d{dt_} L{Lt} n{nt} causal zigzag",
                                "tflops": 3.5 * ff / (statistics.mean(ms) / 1e3) / 1e12,
                                "ms": statistics.mean(ms),
                                "flops": "fwd 4BHL^2d/2 + bwd 2.5x fwd"}
    else:
        res["train_fwd_bwd"] = {"skipped": "backward runs on the CUDA-core path for this shape"}
    fms = time_launches(lambda: ra.fwd(xt["q"], xt["k"], xt["v"], nt, t["causal"], t["layout"],
                                       out=ot, lse=lt, stream=stream), 3, 1, stream)
    res["train_fwd_only"] = {"tflops": ff / (statistics.mean(fms) / 1e3) / 1e12,
                             "ms": statistics.mean(fms)}
    if bwd_steps:  # the backward alone: the step's time less the forward's (both timed above)
        bms = statistics.mean(ms) - statistics.mean(fms)
        res["train_bwd_only"] = {"tflops": 2.5 * ff / (bms / 1e3) / 1e12, "ms": bms,
                                 "frac": 2.5 * ff / (bms / 1e3) / 1e12 / peak_b,
                                 "how": "forward + backward step time minus the forward's, CUDA events"}
    if bwd_steps:  # the same step keeping the forward's float32 output for the backward's D
        o32 = torch.empty(xt["q"].shape, dtype=torch.float32, device=dev)

        def train_step_f32out():
            ra.fwd_f32out(xt["q"], xt["k"], xt["v"], nt, t["causal"], t["layout"], out=o32, lse=lt, stream=stream)
            ra.bwd_f32out(xt["q"], xt["k"], xt["v"], o32, lt, xt["dout"], nt, t["causal"], t["layout"],
                          dq=dq, dk=dk, dv=dv, workspace=wsb, stream=stream)

        ms32 = time_launches(train_step_f32out, bwd_steps, 1, stream)
        res["train_fwd_bwd_f32out"] = {"tflops": 3.5 * ff / (statistics.mean(ms32) / 1e3) / 1e12,
                                       "ms": statistics.mean(ms32),
                                       "what": "ring_attn_fwd_f32out + ring_attn_bwd_f32out (D from the float32 output)"}
        del o32
    del xt, ot, lt, dq, dk, dv, wsb
    # head dim 64 and the striped layout: the long-context forward and the training step
    for name in ("zigzag_gqa_128k_d64", "striped_gqa_128k", "zigzag_gqa_64k_train_d64", "striped_gqa_64k_train"):
        res["workload_" + name] = other_workload(ra, name, stream, dev, peak_b)
    torch.cuda.empty_cache()
    res["device_status"] = ra.device_status()
    return res


if __name__ == "__main__":
    main()
