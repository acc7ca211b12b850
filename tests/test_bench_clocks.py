"""bench.py's host-side helpers: parsing of the nvidia-smi clock samples it
records beside every measurement (no GPU: the sampler's process is faked),
and the oracle's thread count it reports with the CPU baseline."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


class _FakeProc:
    def __init__(self, out):
        self.out = out

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.out, ""


def _sampler(out):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc = _FakeProc(out)
    return s


def test_medians_reasons_and_memory_clock():
    out = ("0, 1575, 2032, 1090.5, 0x4, Not Active, Not Active, Not Active, Active, 3996\n"
           "0, 1560, 2032, 1101.0, 0x4, Not Active, Not Active, Not Active, Active, 3996\n"
           "0, 1590, 2032, 1095.0, 0x0, Not Active, Not Active, Not Active, Not Active, 3996\n")
    c = _sampler(out).stop()
    assert c["sm_mhz"] == 1575.0 and c["sm_max_mhz"] == 2032.0
    assert c["reasons"] == ["sw_power_cap"] and c["samples"] == 3
    assert c["mem_mhz"] == 3996.0 and c["power_w"] == 1095.0


def test_slowdowns_are_reported_and_short_lines_skipped():
    out = ("0, 1200, 2032, 900.0, 0x8, Active, Not Active, Active, Not Active, 3996\n"
           "garbage\n"
           "0, [N/A], 2032\n")
    c = _sampler(out).stop()
    assert c["samples"] == 1
    assert c["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_no_samples_gives_none():
    assert _sampler("").stop() is None
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc = None
    assert s.stop() is None


_HIDE_THREADPOOLCTL = """
import builtins
real = builtins.__import__
def imp(name, *a, **k):
    if name.startswith("threadpoolctl"):
        raise ImportError(name)
    return real(name, *a, **k)
builtins.__import__ = imp
"""


def test_oracle_thread_count_follows_the_blas_pool():
    """`cpu_baseline.cores` reports the oracle's BLAS threads, not the CPU
    count: through threadpoolctl, and without it (from NumPy's own OpenBLAS)."""
    import subprocess
    for prelude in ("", _HIDE_THREADPOOLCTL):
        for n in (1, 3):
            env = dict(os.environ, OPENBLAS_NUM_THREADS=str(n), OMP_NUM_THREADS=str(n))
            code = prelude + "import bench, oracle\nprint(bench.oracle_threads())\n"
            out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                                 timeout=120, check=True).stdout
            assert int(out.strip()) == min(n, len(os.sched_getaffinity(0))), (prelude != "", n, out)
    assert bench.oracle_threads() >= 1
