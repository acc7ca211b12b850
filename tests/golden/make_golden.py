"""Write tests/golden/tiny_decode.txt from the oracle alone.

    python tests/golden/make_golden.py

The fixture records, for the tiny decode workload (batch 1, context 256,
block 16, hidden 256, 4/4 heads x 64, 2 layers, SwiGLU 1024, vocab 4096,
seed 0), the oracle's decode of one block at gamma 0.5 / 0.8 / 0.95
(threshold) and 0.8 (mock-AR): the committed ids, the number of denoising
steps, the commits per step, and the first step's confidences, argmaxes and
near-tie flags.  Only `synth` (inputs) and `oracle` are used.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

CASES = [(0.5, oracle.MODE_THRESHOLD), (0.8, oracle.MODE_THRESHOLD), (0.95, oracle.MODE_THRESHOLD),
         (0.8, oracle.MODE_MOCK_AR)]
PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_decode.txt")


def tiny_model():
    cfg = synth.TINY
    kb, vb = synth.make_context_kv(cfg, 0)
    return oracle.OracleModel.from_bits(cfg, synth.make_weights(cfg, 0), kb, vb, synth.bf16_bits_to_f32)


def decode(model, gamma, mode):
    """One block, stepping the oracle; returns the record written for a case."""
    cfg = model.cfg
    S = cfg.block
    tokens = np.full((1, S), cfg.vocab, np.int32)
    mask = np.full(1, (1 << S) - 1, np.uint32)
    commits, first, any_tie = [], None, False
    while int(mask[0]):
        r = oracle.denoise_step(model, tokens, mask, gamma, mode)
        if first is None:
            first = r
        masked = np.array([(int(mask[0]) >> i) & 1 for i in range(S)], bool)
        any_tie |= bool((r.near_tie[0] & masked).any())
        commits.append(int(r.n_committed[0]))
        tokens, mask = r.tokens, r.mask
        if len(commits) > 4 * S:
            raise RuntimeError("block did not fill")
    return {"tokens": tokens[0].tolist(), "steps": len(commits), "commits": commits,
            "conf": first.conf[0].tolist(), "arg": first.arg[0].tolist(),
            "tie": first.near_tie[0].astype(int).tolist(), "trajectory_tie": int(any_tie)}


def main():
    model = tiny_model()
    lines = ["# Written by tests/golden/make_golden.py from oracle/ (tiny decode workload, seed 0).",
             "# One block of 16 positions per case; first-step values are the oracle's fp32 outputs."]
    for gamma, mode in CASES:
        rec = decode(model, gamma, mode)
        name = "mock_ar" if mode == oracle.MODE_MOCK_AR else "threshold"
        lines.append(f"case gamma={gamma} mode={name} steps={rec['steps']} trajectory_tie={rec['trajectory_tie']}")
        lines.append("tokens " + " ".join(str(t) for t in rec["tokens"]))
        lines.append("commits " + " ".join(str(c) for c in rec["commits"]))
        lines.append("first_conf " + " ".join(f"{c:.9g}" for c in rec["conf"]))
        lines.append("first_arg " + " ".join(str(a) for a in rec["arg"]))
        lines.append("first_tie " + " ".join(str(t) for t in rec["tie"]))
    with open(PATH, "w") as f:
        f.write("\n".join(lines) + "\n")
    print(PATH)


if __name__ == "__main__":
    main()
