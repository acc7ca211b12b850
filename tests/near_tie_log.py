"""Counts of the positions the GPU parity tests waive as near-ties.

The parity bar compares committed ids bit-exactly except at masked
positions the oracle flags as near-ties; every comparison adds its counts
here, and tests/conftest.py prints the totals at the end of the run (also
under -q), so the waived share is visible in every test log."""
from __future__ import annotations

COUNTS: dict[str, list[int]] = {}   # test id -> [flagged positions, masked positions compared]


def record(test_id: str, flagged: int, compared: int) -> None:
    c = COUNTS.setdefault(test_id, [0, 0])
    c[0] += int(flagged)
    c[1] += int(compared)


def summary_lines() -> list[str]:
    if not COUNTS:
        return []
    f = sum(v[0] for v in COUNTS.values())
    n = sum(v[1] for v in COUNTS.values())
    lines = [f"near-tie positions waived by the GPU parity tests: {f} of {n} masked positions compared "
             f"({100.0 * f / max(n, 1):.3f} %)"]
    for k, (a, b) in sorted(COUNTS.items()):
        if a:
            lines.append(f"  {k}: {a} of {b}")
    return lines
