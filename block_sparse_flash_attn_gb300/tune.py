"""Offline sweep of the forward kernel's build-time parameters.

"Pallas-Triton kernels and kernel auto-tuning" (section "Auto-tuning") tunes
a kernel by randomly sampling or exhaustively scanning its parameter space,
compiling each setting and timing it, and prints a table of settings with
their mean and standard deviation.  This is that loop for this library, run
offline (never on the timed path): the kernel's tile is fixed at 128 x 128
by the mask, so the parameters are the ones that are free on GB300:

  BSATTN_EXP2_POLY_PAIRS     of each 32 pairs of exponentials per half row,
                             how many the FMA pipes compute (the rest use MUFU)
  BSATTN_CLAIM_AHEAD         key blocks before a tile's end at which the next
                             tile is claimed and its Q loaded
  BSATTN_SCHED_CHUNK_BLOCKS  key blocks of K/V per schedule chunk (the heads
                             whose tiles run together so their K/V stay in L2)
  BSATTN_D128_QSTAGES / _KSTAGES / _VSTAGES
                             at head_dim 128, the Q buffers and the K and V ring
                             depths (32 KB tiles; at most 7 fit in shared memory)

Each setting is compiled into its own library under _lib/variants/ and timed
by bench.py in a child process (BSATTN_LIBRARY selects the build), on the
given workloads, `repeats` times; the result is a JSON line per (setting,
workload) and a Markdown table sorted by mean time.

  python -m block_sparse_flash_attn_gb300.tune --mode scan --workloads 2,5
  python -m block_sparse_flash_attn_gb300.tune --mode sample --samples 8 --seed 1
"""
from __future__ import annotations

import argparse
import hashlib
import itertools
import json
import os
import random
import statistics
import subprocess
import sys

from . import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# The parameter space: macro -> candidate values (the first is not special;
# the library's defaults are the values compiled in without -D flags).
SPACE = {
    "BSATTN_EXP2_POLY_PAIRS": [0, 2, 4, 6, 8, 10, 12, 14, 16],
    "BSATTN_CLAIM_AHEAD": [2, 4, 6],
    "BSATTN_SCHED_CHUNK_BLOCKS": [384, 768, 1536],
    "BSATTN_D128_QSTAGES": [1, 2],
    "BSATTN_D128_KSTAGES": [2, 3],
    "BSATTN_D128_VSTAGES": [2, 3],
}


def valid(setting: dict) -> bool:
    """Settings the kernel can be built with: at head_dim 128 the Q buffers
    and the K and V stages (32 KB each) fit the 227 KB of shared memory."""
    tiles = sum(setting.get(f"BSATTN_D128_{x}STAGES", d) for x, d in (("Q", 1), ("K", 3), ("V", 3)))
    return tiles <= 7


def settings(space: dict, mode: str, samples: int = 8, seed: int = 0, fixed: dict | None = None):
    """The settings to time, each a dict macro -> value.  scan: every
    combination, in order; sample: `samples` distinct combinations drawn
    uniformly (seeded).  `fixed` pins some macros to one value."""
    space = dict(space)
    for k, v in (fixed or {}).items():
        space[k] = [v]
    keys = sorted(space)
    combos = [dict(zip(keys, vals)) for vals in itertools.product(*(space[k] for k in keys))]
    combos = [c for c in combos if valid(c)]
    if mode == "scan":
        return combos
    if mode != "sample":
        raise ValueError("mode must be 'scan' or 'sample'")
    rng = random.Random(seed)
    return rng.sample(combos, min(samples, len(combos)))


def flags(setting: dict) -> list:
    """nvcc -D flags of one setting."""
    return [f"-D{k}={v}" for k, v in sorted(setting.items())]


def tag(setting: dict) -> str:
    """A short stable name of one setting (its library's directory)."""
    return hashlib.sha1(" ".join(flags(setting)).encode()).hexdigest()[:12]


def parse_bench(stdout: str) -> dict:
    """The bench's one JSON line (the last line that parses as a JSON object)."""
    for line in reversed(stdout.strip().splitlines()):
        line = line.strip()
        if line.startswith("{"):
            try:
                return json.loads(line)
            except json.JSONDecodeError:
                continue
    raise ValueError("no JSON line in the bench output")


def summarize(rows: list) -> list:
    """Per (setting, workload): mean and sample std of the step time (ms) and
    of the throughput over the repeats, sorted by workload then mean time."""
    groups = {}
    for r in rows:
        groups.setdefault((r["tag"], r["workload"]), []).append(r)
    out = []
    for (tg, wl), rs in groups.items():
        ms = [r["ms_per_step"] for r in rs]
        tf = [r["value"] for r in rs]
        out.append({"tag": tg, "workload": wl, "setting": rs[0]["setting"], "n": len(rs),
                    "ms_mean": statistics.mean(ms),
                    "ms_std": statistics.stdev(ms) if len(ms) > 1 else 0.0,
                    "tflops_mean": statistics.mean(tf)})
    out.sort(key=lambda r: (r["workload"], r["ms_mean"]))
    return out


def table(summary: list) -> str:
    """Markdown table of the summary (one block per workload, fastest first)."""
    keys = sorted({k for r in summary for k in r["setting"]})
    head = "| workload | " + " | ".join(k.replace("BSATTN_", "") for k in keys) + \
        " | ms mean | ms std | TFLOP/s |"
    sep = "|" + "---|" * (len(keys) + 4)
    lines = [head, sep]
    for r in summary:
        vals = " | ".join(str(r["setting"][k]) for k in keys)
        lines.append(f"| {r['workload']} | {vals} | {r['ms_mean']:.4f} | {r['ms_std']:.4f} | "
                     f"{r['tflops_mean']:.1f} |")
    return "\n".join(lines)


def run(setting: dict, workloads: list, repeats: int, steps: int, warmup: int) -> list:
    """Build one setting and time it on each workload `repeats` times."""
    lib = os.path.join(_build.LIBDIR, "variants", tag(setting), "libbsattn.so")
    _build.build(extra_flags=flags(setting), out=lib)
    env = dict(os.environ, BSATTN_LIBRARY=lib)
    rows = []
    for w in workloads:
        for rep in range(repeats):
            cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--workload", str(w),
                   "--steps", str(steps), "--warmup", str(warmup), "--configs", "none",
                   "--config-seconds", "0", "--e2e-steps", "0", "--no-cpu-baseline"]
            r = subprocess.run(cmd, capture_output=True, text=True, env=env, cwd=ROOT)
            if r.returncode != 0:
                raise RuntimeError(f"bench failed for {flags(setting)} workload {w}:\n{r.stderr}")
            line = parse_bench(r.stdout)
            rows.append({"tag": tag(setting), "setting": setting, "workload": w, "repeat": rep,
                         "ms_per_step": line["ms_per_step"], "value": line["value"],
                         "clocks": line.get("clocks")})
    return rows


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--mode", default="scan", choices=["scan", "sample"])
    ap.add_argument("--samples", type=int, default=8)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--workloads", default="2,5")
    ap.add_argument("--repeats", type=int, default=3)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--params", default=None,
                    help="comma-separated macros to vary (default: all of SPACE); the others "
                         "keep the library's compiled-in defaults")
    ap.add_argument("--fix", action="append", default=[],
                    help="MACRO=VALUE: hold one parameter at one value")
    ap.add_argument("--out", default=None, help="JSON lines file (default: print only)")
    args = ap.parse_args(argv)
    fixed = {}
    for f in args.fix:
        k, v = f.split("=", 1)
        if k not in SPACE:
            raise SystemExit(f"unknown parameter {k}")
        fixed[k] = int(v)
    wl = [int(x) for x in args.workloads.split(",") if x.strip()]
    space = SPACE
    if args.params:
        names = [x.strip() for x in args.params.split(",") if x.strip()]
        unknown = [x for x in names if x not in SPACE]
        if unknown:
            raise SystemExit(f"unknown parameters {unknown}")
        space = {k: SPACE[k] for k in names}
    rows = []
    for st in settings(space, args.mode, args.samples, args.seed, fixed):
        got = run(st, wl, args.repeats, args.steps, args.warmup)
        rows.extend(got)
        for r in got:
            print(json.dumps(r), flush=True)
            if args.out:
                with open(args.out, "a") as fh:
                    fh.write(json.dumps(r) + "\n")
    print(table(summarize(rows)))


if __name__ == "__main__":
    main()
