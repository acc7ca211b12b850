"""bench.py's multi-rank logic on CPU: two `gloo` ranks on 127.0.0.1.

Each rank decodes its own batch (weak scaling, no collective on the data
path); the bench only reduces its timers: the elapsed time is the max over
ranks and the token count the sum.  The reference arm runs on rank 0 alone.
"""
import contextlib
import io
import json
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    args = bench.parse(["--gpus", str(world), "--impl", "reference", "--config", "tiny", "--steps", "1",
                             "--warmup", "1"])
    w, r, local = bench.dist_setup(args)
    res = {"world": w, "rank": r,
           "max": bench.max_over_ranks(float(rank) + 1.5, w),
           "sum": bench.sum_over_ranks(1.0, w)}
    bench.barrier(w)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(args, w, r)
    res["stdout"] = buf.getvalue()
    import torch.distributed as dist
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(res, f)


def test_two_gloo_ranks(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["world"] == world and d["rank"] == r
        assert d["max"] == 2.5          # max over ranks of rank + 1.5
        assert d["sum"] == 2.0          # tokens add up over ranks
    assert res[1]["stdout"] == ""       # the reference arm prints on rank 0 only
    line = json.loads(res[0]["stdout"].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["n_gpus"] == world and line["scaling"] == "weak"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
