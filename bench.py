#!/usr/bin/env python
"""Benchmark of the block-sparse flash-attention forward on GB300.

Prints ONE JSON line (rank 0):
  metric   effective TFLOP/s over live blocks (4*128*128*D flop per live
           (query block, key block) pair; diagonal causal blocks count in
           full), with its fraction of the bf16 dense tensor peak
  value    whole-job throughput with inputs resident in HBM: sum over ranks of
           live flop / max over ranks of the mean per-step kernel time
  e2e      the same metric through the public API with host buffers
           (HostPipeline): each step copies Q, K, V from pinned host memory to
           the device, runs the forward and copies O and LSE back, all inside
           the timed region; the copies of one piece of the (batch, head)
           range overlap the forward of another
  roofline the forward kernel against the tensor-core peak: achieved =
           live flop per launch / average launch time (CUDA events on the
           launching stream)
  cpu_baseline  the fp64 CPU oracle timed on a bounded sample of the workload

A step is one forward pass (the only kernel of the hot path; the plan is built
once per mask, before the timed region).  L2 is flushed (a 512 MB write)
before every timed step, outside the events.  Inputs are seeded synthetic
tensors (see workloads/).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 1..5]
  python bench.py --impl reference ...   # the oracle as the reference arm
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "bs-attn fwd effective TFLOP/s (live blocks) and % of GB300 BF16 dense peak"
UNIT = "TFLOP/s"
FALLBACK_BF16_TFLOPS = 1900.0   # profiling recipe's fallback (GB300, burst)
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20
# The host-buffer path overlaps pieces of the (batch, head) range: about
# 24 MB of Q, K, V per piece (the upload, ~210 GB/s on the host link, bounds
# the step; smaller pieces shorten the last piece's compute and download).
E2E_PIECE_BYTES = 24 << 20
E2E_MAX_PIECES = 8  # each piece costs a plan, a launch and five copies of host time

# DRAM traffic of one forward launch (dram__bytes_read.sum + dram__bytes_write.sum)
# of the current forward kernel, from the ncu capture summarised in
# profiles/bsattn_fwd_kernel-causal-s4096-d128.md; workloads not captured: None.
TRAFFIC_BYTES = {"w2_bf16": 308_948_736 + 48_557_312}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=2, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--out-f32", action="store_true", help="write O as fp32 (default bf16)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--pass", dest="which", default="fwd", choices=["fwd", "bwd"],
                    help="fwd (default: the forward hot path) or bwd (gradients dQ, dK, dV)")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------
# accounting (host side, from the mask)
# ----------------------------------------------------------------------------

def live_blocks(mask: np.ndarray, causal: bool) -> int:
    m = mask.astype(bool)
    if causal:
        nb = mask.shape[-1]
        m = m & np.tril(np.ones((nb, nb), dtype=bool))
    return int(np.count_nonzero(m))


def flop_per_block(D: int) -> int:
    return 4 * 128 * 128 * D


def row_live_blocks(mask: np.ndarray, causal: bool, rows: np.ndarray, S: int) -> np.ndarray:
    """Live key blocks seen by each flat row id (b*H+h)*S+i."""
    B, H, nb, _ = mask.shape
    bh, i = np.divmod(rows, S)
    qb = i // 128
    m = mask.reshape(B * H, nb, nb)[bh, qb].astype(bool)
    if causal:
        m = m & (np.arange(nb)[None, :] <= qb[:, None])
    return m.sum(axis=1)


def max_over_ranks(x: float, device=None) -> float:
    """Max of a per-rank float over the process group (identity when single-process)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flop_per_rank: float, world: int, ms_max: float) -> float:
    """Units all ranks processed / the slowest rank's time (weak scaling)."""
    return world * flop_per_rank / (ms_max * 1e-3) / 1e12


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        bf16 = d.get("bf16_tflops") or d.get("bf16_tflops_burst")
        return {"bf16": float(bf16), "bf16_sustained": float(d.get("bf16_tflops_sustained", bf16)),
                "hbm": float(d.get("hbm_gbs", FALLBACK_HBM_GBS)), "source": "measured"}
    except Exception:  # noqa: BLE001 - absent or unreadable file
        return {"bf16": FALLBACK_BF16_TFLOPS, "bf16_sustained": 1700.0, "hbm": FALLBACK_HBM_GBS,
                "source": "fallback"}


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:  # noqa: BLE001 - nvidia-smi missing
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ----------------------------------------------------------------------------

def oracle_sample_rate(w, q, k, v, mask, target_s: float, seed: int = 0):
    """Time the oracle on random rows of the workload; returns (TFLOP/s, rows, seconds)."""
    import oracle
    S, D = w.S, w.D
    total_rows = q.shape[0] * q.shape[1] * S
    rng = np.random.default_rng(seed)
    n = 64
    while True:
        rows = np.sort(rng.choice(total_rows, size=min(n, total_rows), replace=False))
        t0 = time.perf_counter()
        oracle.attention(q, k, v, mask, w.scale, w.causal, rows=rows)
        dt = time.perf_counter() - t0
        if dt >= 0.25 * target_s or n >= total_rows:
            break
        n = int(min(total_rows, n * max(2.0, 0.5 * target_s / max(dt, 1e-3))))
    flop = float(row_live_blocks(mask, w.causal, rows, S).sum()) * 128 * 4 * D
    return flop / dt / 1e12, len(rows), dt


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------
# arms
# ----------------------------------------------------------------------------

def run_reference(args):
    w = workloads.WORKLOADS[args.workload]
    q, k, v = workloads.make_qkv(w)
    mask = workloads.make_mask(w)
    per_step = max(1.0, min(6.0, 150.0 / max(1, args.steps + args.warmup)))
    rates, times = [], []
    for i in range(args.warmup + args.steps):
        r, nrows, dt = oracle_sample_rate(w, q, k, v, mask, per_step, seed=i)
        if i >= args.warmup:
            rates.append(r)
            times.append(dt)
    value = float(statistics.mean(rates))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": f"{w.id}:{w.name}", "shape": w.describe(),
                   "sample": "random query rows per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"each step: random query rows of workload {w.id} "
                                   f"(~{per_step:.0f} s of fp64 work), rate over their live keys"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    import torch.distributed as dist

    import block_sparse_flash_attn_gb300 as bsattn
    from block_sparse_flash_attn_gb300 import _build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    _build.build()
    bsattn.load()

    w = workloads.WORKLOADS[args.workload]
    # weak scaling: every rank runs its own full-size problem (independent heads)
    qb, kb, vb = (workloads.normal_bf16(w.data_seed + 100 * rank, s, (w.B, w.H, w.S, w.D), w.mult)
                  for s in (workloads.STREAM_Q, workloads.STREAM_K, workloads.STREAM_V))
    mask = workloads.make_mask(w)
    nlive = live_blocks(mask, w.causal)
    flop = nlive * flop_per_block(w.D)

    def to_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    q, k, v = to_dev(qb), to_dev(kb), to_dev(vb)
    mask_d = torch.from_numpy(mask).to(dev)
    plan = bsattn.plan(mask_d, causal=w.causal, out_f32=args.out_f32)
    o, lse = bsattn.fwd(q, k, v, plan, w.scale)
    bsattn.plan_status(plan)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        flush.zero_()
        bsattn.fwd(q, k, v, plan, w.scale, out=o, lse=lse)
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for s, e in ev:
        flush.zero_()
        s.record(stream)
        bsattn.fwd(q, k, v, plan, w.scale, out=o, lse=lse)
        e.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    bsattn.plan_status(plan)
    ms = [s.elapsed_time(e) for s, e in ev]
    ms_mean = statistics.mean(ms)
    ms_max = max_over_ranks(ms_mean, dev)
    value = whole_job_tflops(flop, world, ms_max)

    # end to end through the public API with pinned host buffers
    hq, hk, hv = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory()
                  for x in (qb, kb, vb))
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    hl = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()

    # the public host-buffer path: per piece of the (batch, head) range, the
    # upload, the forward and the download run on their own streams, overlapped
    pieces = min(w.B * w.H, E2E_MAX_PIECES, max(4, -(-h2d // E2E_PIECE_BYTES)))
    pipe = bsattn.HostPipeline(mask_d, w.D, causal=w.causal, out_f32=args.out_f32,
                               chunks=pieces)

    def e2e_step():
        pipe.run(hq, hk, hv, ho, hl, w.scale, stream=stream)

    e2e_step()
    torch.cuda.synchronize()
    pipe.status()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    pipe.status()
    pipe.close()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, dev)
    e2e_value = whole_job_tflops(flop, world, e2e_ms)

    peaks = read_peaks()
    achieved = flop / (ms_mean * 1e-3) / 1e12
    key = f"w{w.id}_{'f32' if args.out_f32 else 'bf16'}"
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16"], "unit": UNIT,
                "frac": achieved / peaks["bf16"], "traffic": TRAFFIC_BYTES.get(key),
                "peak_source": f"bf16 dense burst, {peaks['source']}",
                "frac_of_spec_2250": achieved / 2250.0,
                "kernel": "bsattn_fwd_kernel", "ms_per_launch": ms_mean}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, nrows, dt = oracle_sample_rate(w, qb, kb, vb, mask, args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{nrows} random query rows of workload {w.id} ({dt:.1f} s, fp64)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"{w.id}:{w.name}", "shape": w.describe(),
                       "out_dtype": "f32" if args.out_f32 else "bf16",
                       "live_blocks": nlive, "flop_per_step": flop,
                       "l2": "flushed (512 MB write) before every timed step",
                       "parallelism": f"replicas x{world} (independent problems, no collective)"},
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": args.steps,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "clocks": clk,
            "wall_s_timed_region": wall,
            "pct_of_peak": 100.0 * value / world / peaks["bf16"],
        }
        print(json.dumps(line), flush=True)
    plan.close()
    if world > 1:
        dist.destroy_process_group()


BWD_METRIC = "bs-attn bwd effective TFLOP/s (live blocks)"


def run_bwd(args):
    """Backward pass: one step = one bsattn_bwd call (the dO.O row term, the
    dK/dV kernel and the dQ kernel) on the workload, inputs resident, L2
    flushed before each."""
    import torch
    import torch.distributed as dist

    import block_sparse_flash_attn_gb300 as bsattn
    from block_sparse_flash_attn_gb300 import _build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    _build.build()
    bsattn.load()

    w = workloads.WORKLOADS[args.workload]
    shape = (w.B, w.H, w.S, w.D)
    qb, kb, vb = (workloads.normal_bf16(w.data_seed + 100 * rank, s, shape, w.mult)
                  for s in (workloads.STREAM_Q, workloads.STREAM_K, workloads.STREAM_V))
    gb = workloads.upstream_grad(w.data_seed + 100 * rank, *shape)
    mask = workloads.make_mask(w)
    nlive = live_blocks(mask, w.causal)
    flop = nlive * 10 * 128 * 128 * w.D  # five 128 x 128 x D products per live block

    def to_dev(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    q, k, v, g = to_dev(qb), to_dev(kb), to_dev(vb), to_dev(gb)
    plan = bsattn.plan(torch.from_numpy(mask).to(dev), causal=w.causal, out_f32=args.out_f32)
    o, lse = bsattn.fwd(q, k, v, plan, w.scale)
    dq, dk, dv = bsattn.bwd(q, k, v, o, lse, g, plan, w.scale)
    bsattn.plan_status(plan)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        flush.zero_()
        bsattn.bwd(q, k, v, o, lse, g, plan, w.scale, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for s, e in ev:
        flush.zero_()
        s.record(stream)
        bsattn.bwd(q, k, v, o, lse, g, plan, w.scale, dq=dq, dk=dk, dv=dv)
        e.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    bsattn.plan_status(plan)
    plan.close()
    ms_mean = statistics.mean(s.elapsed_time(e) for s, e in ev)
    ms_max = max_over_ranks(ms_mean, dev)
    value = whole_job_tflops(flop, world, ms_max)
    peaks = read_peaks()
    achieved = flop / (ms_mean * 1e-3) / 1e12

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and w.S > 8192:
        cpu = {"value": None, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": "skipped: the gradient oracle forms S x S matrices per head "
                         f"(S = {w.S} would need tens of GB)"}
    elif rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        t0 = time.perf_counter()
        oracle.attention_bwd(qb, kb, vb, gb, mask, np.float32(w.scale), w.causal, heads=[(0, 0)])
        dt = time.perf_counter() - t0
        head_flop = live_blocks(mask[:1, :1], w.causal) * 10 * 128 * 128 * w.D
        cpu = {"value": head_flop / dt / 1e12, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"gradients of head (0, 0) of workload {w.id} ({dt:.1f} s, fp64 numpy)"}

    if rank == 0:
        line = {
            "metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"{w.id}:{w.name}", "pass": "bwd", "shape": w.describe(),
                       "grad_dtype": "f32", "live_blocks": nlive, "flop_per_step": flop,
                       "l2": "flushed (512 MB write) before every timed step",
                       "parallelism": f"replicas x{world} (independent problems, no collective)"},
            "e2e": None,
            "gpu_launches": 3 * args.steps,  # row term, dK/dV and dQ kernels
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16"],
                         "unit": UNIT, "frac": achieved / peaks["bf16"], "traffic": None,
                         "peak_source": f"bf16 dense burst, {peaks['source']}",
                         "frac_of_spec_2250": achieved / 2250.0,
                         "kernel": "bsattn_bwd_kernel + bsattn_bwd_dq_kernel + row term "
                                   "(whole step)",
                         "ms_per_launch": ms_mean},
            "cpu_baseline": cpu,
            "clocks": clk,
            "wall_s_timed_region": wall,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main(argv=None):
    args = parse_args(argv)
    if args.which == "bwd":
        if args.impl == "reference":
            raise SystemExit("--pass bwd times the CUDA path only")
        run_bwd(args)
        return
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) == 0:
            run_reference(args)
        return
    run_ours(args)


if __name__ == "__main__":
    main()
