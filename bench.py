#!/usr/bin/env python
"""Benchmark of the block-sparse flash-attention forward on GB300.

Prints ONE JSON line (rank 0):
  metric   effective TFLOP/s over live blocks (4*128*128*D flop per live
           (query block, key block) pair; diagonal causal blocks count in
           full), with its fraction of the bf16 dense tensor peak
  value    whole-job throughput with inputs resident in HBM: sum over ranks of
           live flop / max over ranks of the mean per-step kernel time, on the
           headline workload (default: the random 10 % mask at S = 65536, the
           largest of the five workloads)
  e2e      the same metric through the public API with host buffers
           (HostPipeline): each step copies Q, K, V from pinned host memory to
           the device, runs the forward and copies O and LSE back, all inside
           the timed region; the copies of one piece of the (batch, head)
           range overlap the forward of another
  roofline the forward kernel against its binding roofline: the larger of
           live flop / bf16 tensor peak and algorithmic bytes / HBM peak;
           achieved = that work per launch / average launch time (CUDA events
           on the launching stream); traffic = measured DRAM bytes per launch
           from the committed ncu capture of the same kernel source, else null
  per_config  every one of the five workloads timed the same way for at least
           --config-seconds each (bf16 O), with its own roofline and clocks
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
import dataclasses
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

# Measured DRAM traffic per forward launch: a table under profiles/ written
# from ncu captures (dram__bytes_read.sum + dram__bytes_write.sum), one line
# per (workload, output dtype) with the hash of the kernel source captured.
# A line counts only while the kernel source still has that hash.
TRAFFIC_TABLE = os.path.join(ROOT, "profiles", "bsattn_fwd_kernel-dram-traffic.txt")
KERNEL_SOURCES = [os.path.join(ROOT, "block_sparse_flash_attn_gb300", "csrc", f)
                  for f in ("fwd_sm103.cu", "ptx.cuh", "internal.h")]
HEADLINE_WORKLOAD = 4  # the largest single-GPU workload (B=1 H=32 S=65536 D=128)


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=HEADLINE_WORKLOAD,
                    choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--out-f32", action="store_true", help="write O as fp32 (default bf16)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--e2e-steps", type=int, default=5, help="0 skips the end-to-end leg")
    ap.add_argument("--configs", default="all",
                    help="workloads timed for per_config: 'all', 'none' or a list like 2,5")
    ap.add_argument("--config-seconds", type=float, default=1.0,
                    help="minimum timed seconds per per_config workload")
    ap.add_argument("--heads", type=int, default=None,
                    help="run the workloads with this many heads instead (a smaller case of the "
                         "same kernel, e.g. for an ncu capture)")
    ap.add_argument("--in-dtype", default="bf16", choices=["bf16", "e4m3"],
                    help="e4m3: FP8 Q, K, V (the same normal draws rounded to e4m3; head_dim "
                         "128 workloads only)")
    ap.add_argument("--key-block", type=int, default=128, choices=[128, 64],
                    help="64: the workloads' masks at 64-key granularity (plans with key_block=64)")
    ap.add_argument("--pass", dest="which", default="fwd", choices=["fwd", "bwd"],
                    help="fwd (default: the forward hot path) or bwd (gradients dQ, dK, dV)")
    return ap.parse_args(argv)


# ----------------------------------------------------------------------------
# accounting (host side, from the mask)
# ----------------------------------------------------------------------------

def live_blocks(mask: np.ndarray, causal: bool) -> int:
    """Live (query block, key block) pairs; the key blocks are 128 keys, or 64
    when the mask has twice as many key blocks as query blocks."""
    m = mask.astype(bool)
    if causal:
        nbq, nbk = mask.shape[-2:]
        kdiv = nbk // nbq
        m = m & (np.arange(nbk)[None, :] < kdiv * (np.arange(nbq)[:, None] + 1))
    return int(np.count_nonzero(m))


def allowed_pairs(mask: np.ndarray, causal: bool) -> int:
    """(query, key) pairs the attention actually weighs: every pair of a
    live block, except that under causal a diagonal block (128 x 128, or a
    64-key block that reaches past its query rows) has only its pairs with
    key <= query.  The metric counts whole live blocks; this is the exact
    element count beside it."""
    m = mask.astype(bool)
    nbq, nbk = mask.shape[-2:]
    kdiv = nbk // nbq
    kb = 128 // kdiv
    if not causal:
        return int(np.count_nonzero(m)) * 128 * kb
    qb = np.arange(nbq)[:, None]
    kk = np.arange(nbk)[None, :]
    # allowed pairs of block (qb, kk): query rows 128 qb + r, keys kb * kk + c, c <= ...
    per = np.zeros((nbq, nbk), dtype=np.int64)
    r = np.arange(128)
    for off in range(kdiv):  # key blocks kk = kdiv * qb + off overlap the diagonal
        first_key = kb * off  # relative to the query block's first row
        per_diag = int(np.clip(r[:, None] - (first_key + np.arange(kb))[None, :] + 1, 0, 1).sum())
        per[np.arange(nbq), kdiv * np.arange(nbq) + off] = per_diag
    below = kk < kdiv * qb
    per = np.where(below, 128 * kb, per)
    return int((m * per[None, None]).sum())


def flop_per_block(D: int, key_block: int = 128) -> int:
    return 4 * 128 * key_block * D


def row_live_blocks(mask: np.ndarray, causal: bool, rows: np.ndarray, S: int) -> np.ndarray:
    """Live key blocks seen by each flat row id (b*H+h)*S+i."""
    B, H, nb, nbk = mask.shape
    kdiv = nbk // nb
    bh, i = np.divmod(rows, S)
    qb = i // 128
    m = mask.reshape(B * H, nb, nbk)[bh, qb].astype(bool)
    if causal:
        m = m & (np.arange(nbk)[None, :] < kdiv * (qb[:, None] + 1))
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


def algorithmic_bytes(mask: np.ndarray, causal: bool, S: int, D: int, out_bytes: int,
                      in_bytes: int = 2) -> int:
    """HBM bytes one forward launch cannot avoid: Q rows of tiles with a live
    block, K and V rows of key blocks some tile uses (bf16), O and LSE of every
    row written once, and the plan entries the kernel reads (int32)."""
    B, H, nb, nbk = mask.shape
    kdiv = nbk // nb
    m = mask.astype(bool)
    if causal:
        m = m & (np.arange(nbk)[None, :] < kdiv * (np.arange(nb)[:, None] + 1))
    q_tiles = int(m.any(axis=3).sum())
    kv_blocks = int(m.any(axis=2).sum())
    rows = B * H * S
    plan_words = int(m.sum()) + B * H * nb + 1 + q_tiles
    return (q_tiles * 128 + 2 * kv_blocks * (128 // kdiv)) * D * in_bytes + \
        rows * D * out_bytes + rows * 4 + 4 * plan_words


def roofline(flop: float, nbytes: float, ms: float, peaks: dict, traffic) -> dict:
    """The binding roofline of one launch: the larger of flop / tensor peak and
    algorithmic bytes / HBM peak sets the unit; frac = achieved / peak."""
    t_tensor = flop / (peaks["bf16"] * 1e12)
    t_hbm = nbytes / (peaks["hbm"] * 1e9)
    if t_tensor >= t_hbm:
        achieved = flop / (ms * 1e-3) / 1e12
        r = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16"], "unit": "TFLOP/s",
             "peak_source": f"bf16 dense burst, {peaks['source']}"}
    else:
        achieved = nbytes / (ms * 1e-3) / 1e9
        r = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm"], "unit": "GB/s",
             "peak_source": f"HBM copy bandwidth, {peaks['source']}"}
    r.update(frac=r["achieved"] / r["peak"], traffic=traffic, algorithmic_bytes=nbytes,
             flop=flop, t_floor_us={"tensor": 1e6 * t_tensor, "hbm": 1e6 * t_hbm},
             tflops=flop / (ms * 1e-3) / 1e12, frac_of_spec_2250=flop / (ms * 1e-3) / 1e12 / 2250.0,
             kernel="bsattn_fwd_kernel", ms_per_launch=ms)
    return r


def kernel_source_sha16() -> str:
    """Hash of the forward kernel's source files (which traffic figures apply)."""
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload_id: int, out_f32: bool):
    """DRAM bytes per launch from the committed capture table, if it was taken
    on the current kernel source; else None."""
    want = (str(workload_id), "f32" if out_f32 else "bf16", kernel_source_sha16())
    try:
        with open(TRAFFIC_TABLE) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 5 and not line.startswith("#") and tuple(parts[:3]) == want:
                    return int(parts[3]) + int(parts[4])
    except OSError:
        pass
    return None


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
    kdiv = mask.shape[3] // mask.shape[2]
    total_rows = q.shape[0] * q.shape[1] * S
    rng = np.random.default_rng(seed)
    n = 64
    while True:
        rows = np.sort(rng.choice(total_rows, size=min(n, total_rows), replace=False))
        t0 = time.perf_counter()
        if kdiv == 1:
            oracle.attention(q, k, v, mask, w.scale, w.causal, rows=rows)
        else:
            oracle.attention_kb(q, k, v, mask, w.scale, w.causal, key_block=64, rows=rows)
        dt = time.perf_counter() - t0
        if dt >= 0.25 * target_s or n >= total_rows:
            break
        n = int(min(total_rows, n * max(2.0, 0.5 * target_s / max(dt, 1e-3))))
    flop = float(row_live_blocks(mask, w.causal, rows, S).sum()) * (128 // kdiv) * 4 * D
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


def _workload_list(spec: str, headline: int):
    """per_config workloads in run order, the headline's last (its tensors are
    then reused for the headline's own timed steps)."""
    if spec == "none":
        ids = []
    elif spec == "all":
        ids = sorted(workloads.WORKLOADS)
    else:
        ids = sorted({int(x) for x in spec.split(",") if x.strip()})
    ids = [i for i in ids if i != headline]
    return ids + [headline]


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
    peaks = read_peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    launches = 0

    fp8 = args.in_dtype == "e4m3"
    fwd_call = bsattn.fwd_fp8 if fp8 else bsattn.fwd
    if fp8:  # S = Q K^T at the e4m3 rate (2x bf16), P V in fp16 (1x): half the flop each
        peaks = dict(peaks, bf16=peaks["bf16"] * 4.0 / 3.0,
                     source=f"{peaks['source']} bf16 x 4/3 (e4m3 S, fp16 PV)")

    def to_dev(bits):
        if fp8:
            return torch.from_numpy(bits).to(dev).view(torch.float8_e4m3fn)
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    def traffic_key(wid):
        return f"{wid}" + ("-kb64" if args.key_block == 64 else "") + ("-e4m3" if fp8 else "")

    def launches_per_call(plan, D):
        """Kernel launches of one forward call: where P V runs in fp16 (head_dim
        64, e4m3 inputs) the library may first convert V to fp16 (its plan
        then holds the copy)."""
        return 2 if ((fp8 or D == 64) and bsattn.plan_v16_bytes(plan) > 0) else 1

    def timed(q, k, v, plan, scale, o, lse, steps):
        """steps forward calls, each timed by CUDA events on the launching
        stream after an L2 flush; barrier + synchronize on both sides."""
        nonlocal launches
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for s, e in ev:
            flush.zero_()
            s.record(stream)
            fwd_call(q, k, v, plan, scale, out=o, lse=lse)
            e.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        launches += steps * launches_per_call(plan, q.shape[-1])
        return [s.elapsed_time(e) for s, e in ev], time.perf_counter() - wall0

    def setup(wid, out_f32):
        w = workloads.WORKLOADS[wid]
        if args.heads:
            w = dataclasses.replace(w, H=args.heads)
        # weak scaling: every rank runs its own full-size problem (independent heads)
        gen = workloads.normal_e4m3 if fp8 else workloads.normal_bf16
        bits = tuple(gen(w.data_seed + 100 * rank, st, (w.B, w.H, w.S, w.D), w.mult)
                     for st in (workloads.STREAM_Q, workloads.STREAM_K, workloads.STREAM_V))
        mask = workloads.make_mask(w) if args.key_block == 128 else workloads.make_mask_kb64(w)
        q, k, v = (to_dev(b) for b in bits)
        mask_d = torch.from_numpy(mask).to(dev)
        plan = bsattn.plan(mask_d, causal=w.causal, out_f32=out_f32, key_block=args.key_block)
        o, lse = fwd_call(q, k, v, plan, w.scale)
        bsattn.plan_status(plan)
        return w, bits, mask, mask_d, q, k, v, plan, o, lse

    # ---- per_config: every workload for at least --config-seconds; the
    # headline workload last, its clock record running on into the headline steps
    per_config = {}
    head = None
    head_clock = None
    if fp8 and workloads.WORKLOADS[args.workload].D != 128:
        raise SystemExit("--in-dtype e4m3 takes a head_dim 128 workload (2, 3 or 4)")
    for wid in _workload_list(args.configs, args.workload):
        if fp8 and workloads.WORKLOADS[wid].D != 128:
            continue  # e4m3 inputs at head_dim 128 only
        is_head = wid == args.workload
        out_f32 = args.out_f32 if is_head else False
        w, bits, mask, mask_d, q, k, v, plan, o, lse = setup(wid, out_f32)
        for _ in range(max(3, args.warmup)):
            flush.zero_()
            fwd_call(q, k, v, plan, w.scale, out=o, lse=lse)
        est, _ = timed(q, k, v, plan, w.scale, o, lse, 3)
        est_ms = statistics.mean(est)
        steps_c = int(min(4000, max(args.steps, np.ceil(1e3 * args.config_seconds /
                                                         max(est_ms, 1e-3)))))
        clocks = ClockSampler(local)
        clocks.start()
        ms, wall = timed(q, k, v, plan, w.scale, o, lse, steps_c)
        bsattn.plan_status(plan)
        nlive = live_blocks(mask, w.causal)
        flop = nlive * flop_per_block(w.D, args.key_block)
        ms_max = max_over_ranks(statistics.mean(ms), dev)
        nbytes = algorithmic_bytes(mask, w.causal, w.S, w.D, 4 if out_f32 else 2,
                                   1 if fp8 else 2)
        entry = {"workload": f"{w.id}:{w.name}", "out_dtype": "f32" if out_f32 else "bf16",
                 "flop_elementwise": allowed_pairs(mask, w.causal) * 4 * w.D,
                 "steps": steps_c, "ms_per_step": ms_max,
                 "value": whole_job_tflops(flop, world, ms_max), "unit": UNIT,
                 "wall_s_timed_region": wall,
                 "roofline": roofline(flop, nbytes, statistics.mean(ms), peaks,
                                      measured_traffic(traffic_key(w.id), out_f32))}
        if is_head:
            head = (w, bits, mask, mask_d, q, k, v, plan, o, lse, nlive, flop, nbytes)
            head_clock = clocks
        else:
            entry["clocks"] = clocks.stop()
            plan.close()
            del q, k, v, o, lse, mask_d
        per_config[str(wid)] = entry

    # ---- headline: exactly --steps timed steps after --warmup untimed ones
    w, bits, mask, mask_d, q, k, v, plan, o, lse, nlive, flop, nbytes = head
    for _ in range(args.warmup):
        flush.zero_()
        fwd_call(q, k, v, plan, w.scale, out=o, lse=lse)
    torch.cuda.synchronize()
    ms, wall = timed(q, k, v, plan, w.scale, o, lse, args.steps)
    head_launches = args.steps * launches_per_call(plan, q.shape[-1])
    clk = head_clock.stop()
    if str(w.id) in per_config:
        per_config[str(w.id)]["clocks"] = clk
    bsattn.plan_status(plan)
    ms_mean = statistics.mean(ms)
    ms_max = max_over_ranks(ms_mean, dev)
    value = whole_job_tflops(flop, world, ms_max)

    # ---- end to end through the public API with pinned host buffers
    e2e = None
    # the host pipeline takes bf16 inputs and 128-key blocks
    if args.e2e_steps > 0 and args.key_block == 128 and not fp8:
        qb, kb, vb = bits
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
        pipe.run(hq, hk, hv, ho, hl, w.scale, stream=stream)
        torch.cuda.synchronize()
        pipe.status()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            pipe.run(hq, hk, hv, ho, hl, w.scale, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        pipe.status()
        pipe.close()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, dev)
        e2e = {"value": whole_job_tflops(flop, world, e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "pieces": pieces}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        if fp8:  # the oracle on the decoded inputs (the same fp64 work)
            import oracle
            bits = tuple(np.ascontiguousarray(oracle.decode_e4m3(b)) for b in bits)
        rate, nrows, dt = oracle_sample_rate(w, *bits, mask, args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{nrows} random query rows of workload {w.id} ({dt:.1f} s, fp64)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if fp8 else "bf16",
            "data": "synthetic",
            "config": {"workload": f"{w.id}:{w.name}", "shape": w.describe(args.in_dtype),
                       "out_dtype": "f32" if args.out_f32 else "bf16",
                       "key_block": args.key_block, "in_dtype": args.in_dtype,
                       "live_blocks": nlive, "flop_per_step": flop,
                       "flop_elementwise": allowed_pairs(mask, w.causal) * 4 * w.D,
                       "l2": "flushed (512 MB write) before every timed step",
                       "parallelism": f"replicas x{world} (independent problems, no collective)"},
            "e2e": e2e,
            "gpu_launches": head_launches,
            "roofline": roofline(flop, nbytes, ms_mean, peaks,
                                 measured_traffic(traffic_key(w.id), args.out_f32)),
            "cpu_baseline": cpu,
            "clocks": clk,
            "clocks_note": "sampled from the start of this workload's per_config timing "
                           "through the end of the headline steps",
            "wall_s_timed_region": wall,
            "pct_of_peak": 100.0 * value / world / peaks["bf16"],
            "kernel_source_sha16": kernel_source_sha16(),
            "per_config": per_config,
            "gpu_launches_all_timed_regions": launches,
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
            "gpu_launches": 2 * args.steps,  # row term; dK/dV and dQ in one launch
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
