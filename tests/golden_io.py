"""Readers for the text fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _kv(tokens):
    return dict(t.split("=", 1) for t in tokens)


def mode_code(name: str) -> int:
    """threshold | mock_ar | topk:k | steps:N -> the library's mode value."""
    if name in ("threshold", "mock_ar"):
        return 0 if name == "threshold" else 1
    kind, _, val = name.partition(":")
    return {"topk": 2, "steps": 3}[kind] | (int(val) << 8)


def commit_cases():
    """Yield dicts: name, gamma, mode (0 threshold / 1 mock-AR), mask, conf [16],
    committed (list of positions), mask_after."""
    lines = [l.strip() for l in open(os.path.join(GOLDEN, "commit_rule.txt")) if l.strip() and not l.startswith("#")]
    for i in range(0, len(lines), 3):
        head, conf, expect = lines[i].split(), lines[i + 1].split(), lines[i + 2].split()
        assert head[0] == "case" and conf[0] == "conf" and expect[0] == "expect"
        h, e = _kv(head[2:]), _kv(expect[1:])
        yield {"name": head[1], "gamma": float(h["gamma"]), "mode": mode_code(h["mode"]),
               "mask": int(h["mask"], 16), "conf": np.array([float(v) for v in conf[1:]], np.float32),
               "committed": [] if e["committed"] == "-" else [int(v) for v in e["committed"].split(",")],
               "mask_after": int(e["mask"], 16)}


def tiny_decode_cases():
    """Yield dicts: gamma, mode, steps, trajectory_tie, tokens, commits,
    first_conf, first_arg, first_tie."""
    lines = [l.split() for l in open(os.path.join(GOLDEN, "tiny_decode.txt")) if l.strip() and not l.startswith("#")]
    for i in range(0, len(lines), 6):
        h = _kv(lines[i][1:])
        rec = {"gamma": float(h["gamma"]), "mode": 1 if h["mode"] == "mock_ar" else 0, "steps": int(h["steps"]),
               "trajectory_tie": bool(int(h["trajectory_tie"]))}
        for row in lines[i + 1:i + 6]:
            key, vals = row[0], row[1:]
            rec[key] = np.array([float(v) for v in vals], np.float32) if key == "first_conf" else \
                np.array([int(v) for v in vals], np.int64)
        yield rec


def near_tie_cases():
    """Yield dicts: name, gamma, mode, mask, conf [16] fp32, gap [16], flagged
    (list of positions); the logit row of position i is [0, -gap_i, -20, -20]."""
    lines = [l.strip() for l in open(os.path.join(GOLDEN, "near_tie_cases.txt")) if l.strip() and not l.startswith("#")]
    for i in range(0, len(lines), 4):
        head, conf, gap, expect = (lines[i + j].split() for j in range(4))
        assert head[0] == "case" and conf[0] == "conf" and gap[0] == "gap" and expect[0] == "expect"
        h, e = _kv(head[2:]), _kv(expect[1:])
        yield {"name": head[1], "gamma": float(h["gamma"]), "mode": mode_code(h["mode"]),
               "mask": int(h["mask"], 16), "conf": np.array([float(v) for v in conf[1:]], np.float32),
               "gap": np.array([float(v) for v in gap[1:]], np.float32),
               "flagged": [] if e["flagged"] == "-" else [int(v) for v in e["flagged"].split(",")]}


def near_tie_logits(gap):
    """Logit rows [0, -gap_i, -20, -20] (fp32) whose top-2 gap is gap_i."""
    g = np.asarray(gap, np.float32)
    rows = np.full((g.size, 4), -20.0, np.float32)
    rows[:, 0] = 0.0
    rows[:, 1] = -g
    return rows
