"""Committed tokens/s for every decode workload, gamma and commit mode.

    python -m block_wise_masked_dd_b300.sweep [--configs tiny small large] [--steps K] [--warmup W]
                                              [--modes mock_ar topk:2 steps:8]

Runs `bench.py` once per (workload, gamma, mode) in a fresh process (so each
measurement sees a fresh context and its own clock record), and prints one
JSON line per run followed by a markdown table.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GAMMAS = (0.5, 0.8, 0.95)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--configs", nargs="+", default=["tiny", "small", "large"])
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--modes", nargs="+", default=["mock_ar", "topk:2", "steps:8"],
                    help="commit modes run besides the threshold rule at each gamma")
    ap.add_argument("--extras", action="store_true",
                    help="also gamma 0.8 with the context grown by the context tower, and with RoPE positions")
    args = ap.parse_args()
    rows = []
    for cfg in args.configs:
        runs = [(g, "threshold", []) for g in GAMMAS] + [(0.8, m, []) for m in args.modes]
        if args.extras:
            runs += [(0.8, "threshold", ["--context-tower"]), (0.8, "threshold", ["--rope-theta", "10000"])]
        for gamma, mode, extra in runs:
            cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--config", cfg, "--gamma", str(gamma), "--mode",
                   mode, "--steps", str(args.steps), "--warmup", str(args.warmup), "--no-micro", "--no-cpu", "--no-small", *extra]
            out = subprocess.run(cmd, capture_output=True, text=True, cwd=ROOT)
            if out.returncode != 0:
                print(json.dumps({"config": cfg, "gamma": gamma, "mode": mode, "error": out.stderr[-2000:]}))
                continue
            line = json.loads(out.stdout.strip().splitlines()[-1])
            print(json.dumps(line), flush=True)
            rows.append((cfg, gamma, mode + (" " + " ".join(extra) if extra else ""), line))
    print("\n| workload | gamma | mode | steps/block | committed tokens/s | e2e tokens/s | ms per bench step | "
          "SM MHz | throttle |")
    print("|---|---|---|---|---|---|---|---|---|")
    for cfg, gamma, mode, l in rows:
        c = l.get("clocks") or {}
        print(f"| {cfg} | {gamma} | {mode} | {l['config']['denoise_steps_per_block']:.2f} | {l['value']:.0f} | "
              f"{l['e2e']['value']:.0f} | {l['ms_per_step']:.2f} | {c.get('sm_mhz', 'n/a')} | "
              f"{','.join(c.get('reasons', [])) or 'none'} |")


if __name__ == "__main__":
    main()
