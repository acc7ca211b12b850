"""Benchmark: committed tokens/s of block-wise masked-diffusion decoding on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config small|tiny|large] [--gamma 0.8] [--mode threshold|mock_ar]

One step = one pass of the whole hot path over one batch: the decode of 8
consecutive 16-position blocks for every sequence of the batch (each block
runs denoising steps until no position is masked; after each block the
context grows by 16 fresh K/V positions, standing in for the frozen context
tower encoding the committed block).  Inputs are synthetic and seeded (random
weights; no datasets or trained checkpoints exist here).

Prints ONE JSON line (rank 0).  Under torchrun each rank decodes its own
batch on its own GPU (weak scaling, no collective on the data path); the
reported time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

BLOCKS_PER_STEP = 8
METRIC = "committed tokens/sec on 1 B300 (block 16, γ=0.8); block-attn HBM GB/s vs peak"
UNIT = "tokens/s"


def mode_arg(s: str) -> str:
    if s in ("threshold", "mock_ar"):
        return s
    name, _, val = s.partition(":")
    if name in ("topk", "steps") and val.isdigit() and 1 <= int(val) <= 65535:
        return s
    raise argparse.ArgumentTypeError(f"bad mode {s!r}")


def mode_code(s: str) -> int:
    """The library's mode value for a --mode string."""
    if s == "threshold":
        return 0
    if s == "mock_ar":
        return 1
    name, _, val = s.partition(":")
    return (2 if name == "topk" else 3) | (int(val) << 8)


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="small", choices=["tiny", "small", "large"])
    ap.add_argument("--gamma", type=float, default=0.8)
    ap.add_argument("--mode", default="threshold", type=mode_arg,
                    help="threshold | mock_ar | topk:K (the K most confident) | steps:N (fixed N steps per block)")
    ap.add_argument("--rope-theta", type=float, default=0.0,
                    help="rotary positions on the block's queries and keys (0: learned in-block positions only)")
    ap.add_argument("--context-tower", action="store_true",
                    help="append each decoded block to the context with the synthetic context tower on the device "
                         "(default: fresh seeded K/V from the host)")
    ap.add_argument("--fused-reduce", action="store_true",
                    help="linear layers reduce their split-K partials inside the GEMM (groups of CTAs) "
                         "instead of in separate kernels (the default)")
    ap.add_argument("--no-micro", action="store_true", help="skip the attention / LM-head microbenchmarks")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    return ap.parse_args(argv)


def workload_desc(cfg, gamma, mode, tower=False):
    return (f"{cfg.name} decode: batch {cfg.batch}, context {cfg.ctx_len} (+16 per block, "
            f"{BLOCKS_PER_STEP} consecutive blocks), block {cfg.block}, hidden {cfg.hidden}, "
            f"{cfg.n_q_heads} q / {cfg.n_kv_heads} kv heads x d{cfg.head_dim}, {cfg.n_layers} layers, "
            f"SwiGLU {cfg.mlp}, vocab {cfg.vocab}, gamma {gamma}, {mode}"
            + (f", RoPE theta {cfg.rope_theta:g}" if cfg.rope_theta > 0 else "")
            + (", context grown on the device by the context tower" if tower else ""))


def bench_cfg(name, rope_theta=0.0):
    cfg = synth.CONFIGS[name]
    return cfg.replace(max_ctx=cfg.ctx_len + BLOCKS_PER_STEP * cfg.block, rope_theta=rope_theta)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6400.0, 1800.0, 1400.0, "fallback"


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------- CPU arm

def oracle_block_sample(cfg, gamma, mode, seed=0, batch=None):
    """Decode one block with the oracle on `batch` sequences of the workload;
    returns (committed tokens, seconds, threads)."""
    import oracle
    c = cfg if batch is None else cfg.replace(batch=batch)
    wb = synth.make_weights(c, seed)
    kb, vb = synth.make_context_kv(c, seed)
    m = oracle.OracleModel.from_bits(c, wb, kb, vb, synth.bf16_bits_to_f32)
    t0 = time.perf_counter()
    tok, steps, _ = oracle.decode_block(m, gamma, mode_code(mode))
    dt = time.perf_counter() - t0
    return c.batch * c.block, dt, os.cpu_count()


def run_reference(args, world, rank):
    cfg = bench_cfg(args.config, args.rope_theta)
    if rank != 0:
        return
    import oracle
    sample_b = 1 if cfg.name != "tiny" else cfg.batch
    c = cfg.replace(batch=sample_b)
    wb = synth.make_weights(c, 0)
    kb, vb = synth.make_context_kv(c, 0)
    m = oracle.OracleModel.from_bits(c, wb, kb, vb, synth.bf16_bits_to_f32)
    mode = mode_code(args.mode)
    for _ in range(args.warmup):
        oracle.decode_block(m, args.gamma, mode)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode_block(m, args.gamma, mode)
    dt = time.perf_counter() - t0
    tokens = args.steps * c.batch * c.block
    value = tokens / dt
    sample = (f"oracle (NumPy fp32, {os.cpu_count()} host threads) decoding one 16-position block of "
              f"{c.batch} sequence(s) of the {cfg.name} workload per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": workload_desc(cfg, args.gamma, args.mode), "tokens_per_step": c.batch * c.block,
                       "parallelism": f"host cores ({os.cpu_count()} threads), rank 0 only",
                       "sample": f"{c.batch} sequence(s) of the workload, one block per step"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch, from
# one ncu capture of the same kernel at the same workload; kinds and workloads
# not captured report null.
TRAFFIC = {("small", "gemm_gate_up"): 47.23e6 + 0.33e6}


def algorithmic_bytes(cfg, kind, ctx_len):
    """Minimum HBM bytes of one launch of `kind` (weights/KV read once,
    activations in and out at their stored precision)."""
    R, H, F, V = cfg.rows, cfg.hidden, cfg.mlp, cfg.vocab
    HqD, qkvw = cfg.n_q_heads * cfg.head_dim, cfg.qkv_width
    if kind == "gemm_qkv":
        return 2 * (qkvw * H + R * H + R * qkvw)
    if kind == "gemm_o":
        return 2 * (H * HqD + R * HqD + R * H)
    if kind == "gemm_gate_up":
        return 2 * (2 * F * H + R * H + R * 2 * F)
    if kind == "gemm_down":
        return 2 * (H * F + R * F + R * H)
    if kind == "lm_head_select":
        return 2 * (V * H + R * H) + 12 * R
    if kind == "attention_context":
        return 2 * 2 * cfg.batch * cfg.n_kv_heads * ctx_len * cfg.head_dim + 2 * R * (qkvw + HqD)
    return None


def mlp_gemm_rates(cfg, kernels, hbm_peak, tc_sust, peak_src):
    """The MLP GEMMs (gate|up, down) of the step from the per-kind profile: HBM
    rate of their algorithmic bytes, and tensor rate of their algorithmic
    FLOPs (2*R*K*N) and of the FLOPs the tensor cores execute (twice that: the
    activation operand is a bf16 head plus a bf16 remainder), against the
    sustained bf16 peak (kernels timed inside a long step)."""
    R, H, F = cfg.rows, cfg.hidden, cfg.mlp
    out = {}
    for kind, n, k in (("gemm_gate_up", 2 * F, H), ("gemm_down", H, F)):
        if kind not in kernels:
            continue
        us = kernels[kind]["us_per_launch"]
        flops = 2.0 * R * k * n
        tf = flops / (us * 1e-6) / 1e12
        gbs = algorithmic_bytes(cfg, kind, 0) / (us * 1e-6) / 1e9
        out[kind] = {"us_per_launch": us, "hbm_GBps": gbs, "hbm_frac": gbs / hbm_peak,
                     "tflops_algorithmic": tf, "tflops_executed": 2 * tf, "tensor_peak_tflops": tc_sust,
                     "tensor_frac_algorithmic": tf / tc_sust, "tensor_frac_executed": 2 * tf / tc_sust,
                     "peak_source": peak_src + " (sustained bf16)"}
    return out


def step_roofline(cfg, T0, hbm_peak, ms_per_step, denoise_per_step, peak_src):
    """The whole denoising step against HBM: every weight read once, the context
    K/V of every layer read once (mean context over the step's blocks)."""
    H, F, V, L = cfg.hidden, cfg.mlp, cfg.vocab, cfg.n_layers
    HqD = cfg.n_q_heads * cfg.head_dim
    weights = 2 * (L * (cfg.qkv_width * H + H * HqD + 2 * F * H + H * F) + V * H)
    t_mean = T0 + cfg.block * (BLOCKS_PER_STEP - 1) / 2
    kv = 2 * 2 * L * cfg.batch * cfg.n_kv_heads * t_mean * cfg.head_dim
    ideal_us = (weights + kv) / (hbm_peak * 1e9) * 1e6
    measured_us = 1e3 * ms_per_step / max(denoise_per_step, 1e-9)
    return {"bytes_per_denoising_step": weights + kv, "ideal_us": ideal_us, "measured_us": measured_us,
            "frac": ideal_us / measured_us, "peak_GBps": hbm_peak, "peak_source": peak_src}


def gpu_arm(args, world, rank, local):
    import torch

    from block_wise_masked_dd_b300 import binding as B
    from block_wise_masked_dd_b300 import build as libbuild
    from block_wise_masked_dd_b300.decoder import BlockAttention, Decoder, LmHeadSelect, pack_weights

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    libbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = bench_cfg(args.config, args.rope_theta)
    mode = mode_code(args.mode)
    hbm_peak, tc_peak, tc_sust, peak_src = load_peaks()

    # weights: the same replica on every rank; context differs per rank
    if cfg.name == "large":
        w = synth.make_weights_torch(cfg, 0, dev)
        k0, v0 = synth.make_context_kv_torch(cfg, 1 + rank, dev)
    else:
        w = synth.make_weights(cfg, 0)
        kb, vb = synth.make_context_kv(cfg, rank)
        from block_wise_masked_dd_b300.decoder import bits_to_tensor
        k0, v0 = bits_to_tensor(kb, dev), bits_to_tensor(vb, dev)
    weights = pack_weights(cfg, w, dev)
    del w
    dec = Decoder(cfg, weights, dev)
    if args.fused_reduce:
        dec.fused_reduce = True
    if dec.fused_reduce:
        linear = "split-K reduced in the GEMM by groups of " + ", ".join(
            f"{k} {cs}" for k, (cs, _) in dec.fused_plan().items())
    else:
        linear = "split-K partials reduced by separate kernels"
    T0 = cfg.ctx_len
    dec.set_context_kv(k0, v0, 0)
    del k0, v0
    # appended context K/V per block: device copies and pinned host copies (e2e)
    gen = synth.torch_generator(100 + rank, dev)
    app_shape = (cfg.n_layers, cfg.batch, cfg.n_kv_heads, cfg.block, cfg.head_dim)
    app = [(synth.torch_normal_bf16(app_shape, 1.0, gen, dev), synth.torch_normal_bf16(app_shape, 1.0, gen, dev))
           for _ in range(BLOCKS_PER_STEP)]
    app_host = [(k.cpu().pin_memory(), v.cpu().pin_memory()) for k, v in app]
    tokens = torch.empty((BLOCKS_PER_STEP, cfg.batch, cfg.block), dtype=torch.int32, device=dev)
    tokens_host = torch.empty((BLOCKS_PER_STEP, cfg.batch, cfg.block), dtype=torch.int32).pin_memory()
    stream = torch.cuda.current_stream(dev)
    per_step_launches = B.dd_step_launch_count(dec.ctx)
    counters = {"denoise_steps": 0, "launches": 0}

    if args.context_tower:
        tw = (synth.make_tower_weights_torch(cfg, 0, dev) if cfg.name == "large" else synth.make_tower_weights(cfg, 0))
        dec.set_context_tower(tw)
        del tw

    def one_step(host: bool):
        dec.set_context_len(T0)
        counters["launches"] += 1
        for blk in range(BLOCKS_PER_STEP):
            if args.context_tower:
                # the committed block goes to the context on the device; the
                # host only reads the committed ids
                _, steps = dec.decode_block(args.gamma, mode, tokens=tokens[blk])
                dec.append_block(tokens[blk])
                if host:
                    tokens_host[blk].copy_(tokens[blk], non_blocking=True)
                counters["launches"] += 3 + steps * per_step_launches + 3  # + embed, GEMM, reduce-append
            else:
                out = tokens_host[blk] if host else tokens[blk]
                _, steps = dec.decode_block(args.gamma, mode, tokens=out)
                k, v = app_host[blk] if host else app[blk]
                dec.set_context_kv(k, v, T0 + blk * cfg.block)
                counters["launches"] += 3 + steps * per_step_launches + 1  # block init, params, loop init; length
            counters["denoise_steps"] += steps

    # ---------------------------------------------------- timed region
    for _ in range(args.warmup):
        one_step(False)
    torch.cuda.synchronize(dev)
    barrier(world)
    counters.update(denoise_steps=0, launches=0)
    clocks = ClockSampler(local)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    for _ in range(args.steps):
        one_step(False)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    barrier(world)
    ms = ev0.elapsed_time(ev1)
    timed_denoise = counters["denoise_steps"]
    timed_launches = counters["launches"]
    ms_max = max_over_ranks(ms, world)
    tokens_per_step = cfg.batch * cfg.block * BLOCKS_PER_STEP
    total_tokens = sum_over_ranks(tokens_per_step * args.steps, world)
    value = total_tokens / (ms_max / 1e3)

    # ---------------------------------------------- end to end (host buffers)
    counters.update(denoise_steps=0, launches=0)
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step(True)
    torch.cuda.synchronize(dev)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    e2e_value = total_tokens / e2e_s
    h2d = 0 if args.context_tower else BLOCKS_PER_STEP * 2 * app_host[0][0].numel() * 2
    d2h = tokens_per_step * 4

    # ------------------------------------- per-kernel profile of the step
    prof = {}
    t_, m_ = (torch.full((cfg.batch, cfg.block), cfg.vocab, dtype=torch.int32, device=dev),
              torch.full((cfg.batch,), (1 << cfg.block) - 1, dtype=torch.int32, device=dev))
    dec.set_context_len(T0)
    nprof = 0
    commits = []  # positions committed per denoising step of the first block (all sequences)

    def masked_count():
        return int(sum(bin(int(v) & 0xFFFFFFFF).count("1") for v in m_.cpu().tolist()))
    left = masked_count()
    while left and nprof < 4 * cfg.block:
        for kind, msk in B.dd_profile_step(dec.ctx, t_.data_ptr(), m_.data_ptr(), args.gamma, mode,
                                           stream=stream.cuda_stream):
            p = prof.setdefault(kind, [0.0, 0])
            p[0] += msk
            p[1] += 1
        nprof += 1
        now = masked_count()
        commits.append(left - now)
        left = now
    total_prof = sum(v[0] for v in prof.values())
    kernels = {k: {"launches": v[1], "ms_total": v[0], "share": v[0] / total_prof,
                   "us_per_launch": 1e3 * v[0] / v[1]} for k, v in prof.items()}
    dom = max(prof, key=lambda k: prof[k][0])
    dom_bytes = algorithmic_bytes(cfg, dom, T0)
    dom_us = 1e3 * prof[dom][0] / prof[dom][1]
    roofline = None
    if dom_bytes is not None:
        ach = dom_bytes / (dom_us * 1e-6) / 1e9
        roofline = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
                    "frac": ach / hbm_peak, "traffic": TRAFFIC.get((cfg.name, dom)), "peak_source": peak_src,
                    "algorithmic_bytes_per_launch": dom_bytes, "us_per_launch": dom_us}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_desc(cfg, args.gamma, args.mode, args.context_tower),
                       "tokens_per_step": tokens_per_step, "parallelism": f"dp{world} (independent batches)",
                       "denoise_steps_per_block": timed_denoise / (args.steps * BLOCKS_PER_STEP),
                       "linear_layers": linear,
                       "l2": "inputs larger than L2 (weights + context K/V per denoising step exceed 126 MB)"},
            "gpu_launches": timed_launches, "clocks": clk,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "roofline": roofline, "kernels": kernels,
            "commits_per_step": {"first_block": commits, "mean": float(np.mean(commits)) if commits else None},
            "step_roofline": step_roofline(cfg, T0, hbm_peak, ms_max / args.steps,
                                           timed_denoise / max(args.steps, 1), peak_src),
            "mlp_gemms": mlp_gemm_rates(cfg, kernels, hbm_peak, tc_sust, peak_src)}

    # -------------------------------- microbenchmarks named by the metric
    if not args.no_micro and rank == 0:
        line["attn_microbench"] = attn_micro(dev, stream, hbm_peak, peak_src)
        line["lmhead_microbench"] = lmhead_micro(dev, stream, tc_peak, peak_src)
    if not args.no_cpu and rank == 0:
        n, dt, cores = oracle_block_sample(cfg, args.gamma, args.mode)
        line["cpu_baseline"] = {"value": n / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"one 16-position block of all {cfg.batch} sequences of the "
                                          f"{cfg.name} workload at gamma {args.gamma}, {dt:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    dec.close()


def _time_launches(fn, stream, n):
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / n


def attn_micro(dev, stream, hbm_peak, peak_src):
    """Block attention, batch 64 x context 8192, 32/8 heads x 128 (inputs 2.2 GB > L2)."""
    import torch
    from block_wise_masked_dd_b300.decoder import BlockAttention
    c = synth.ATTN_MICRO
    g = synth.torch_generator(7, dev)
    qkv = synth.torch_normal_bf16((c.rows, c.qkv_width), 1.0, g, dev)
    kc = synth.torch_normal_bf16((c.batch, c.n_kv_heads, c.ctx_len, c.head_dim), 1.0, g, dev)
    vc = synth.torch_normal_bf16((c.batch, c.n_kv_heads, c.ctx_len, c.head_dim), 1.0, g, dev)
    out = torch.empty((c.rows, c.n_q_heads * c.head_dim), dtype=torch.bfloat16, device=dev)
    op = BlockAttention(c.batch, c.block, c.n_q_heads, c.n_kv_heads, c.head_dim, c.ctx_len, c.ctx_len, dev)
    ms = _time_launches(lambda: op(qkv, kc, vc, out, stream), stream, 20)
    nbytes = 2 * 2 * c.batch * c.n_kv_heads * c.ctx_len * c.head_dim + 2 * c.rows * (c.qkv_width + c.n_q_heads * c.head_dim)
    flops = 4 * c.head_dim * c.rows * c.n_q_heads * (c.ctx_len + c.block)
    ach = nbytes / (ms * 1e-3) / 1e9
    del qkv, kc, vc, out
    return {"workload": "block attention: batch 64, context 8192, block 16, 32 q / 8 kv heads x 128",
            "us_per_launch": ms * 1e3, "bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
            "frac": ach / hbm_peak, "peak_source": peak_src, "algorithmic_bytes_per_launch": nbytes,
            "tflops": flops / (ms * 1e-3) / 1e12}


def lmhead_micro(dev, stream, tc_peak, peak_src):
    """LM head + select, 1024 rows x 4096 x 131072 (weights 1.07 GB > L2)."""
    import torch
    from block_wise_masked_dd_b300.decoder import LmHeadSelect
    rows, H, V = 1024, 4096, 131072
    g = synth.torch_generator(9, dev)
    x = synth.torch_normal_bf16((rows, H), 1.0, g, dev)
    w = synth.torch_normal_bf16((V, H), synth.LOGIT_STD / np.sqrt(H), g, dev)
    conf = torch.empty(rows, dtype=torch.float32, device=dev)
    arg = torch.empty(rows, dtype=torch.int32, device=dev)
    op = LmHeadSelect(rows, H, V, dev)
    ms = _time_launches(lambda: op(x, w, conf, arg, stream), stream, 10)
    flops = 2.0 * rows * H * V
    ach = flops / (ms * 1e-3) / 1e12
    del x, w
    return {"workload": "LM head + confidence select: 1024 rows x hidden 4096 x vocab 131072",
            "us_per_launch": ms * 1e3, "bound": "tensor", "achieved": ach, "peak": tc_peak, "unit": "TFLOP/s",
            "frac": ach / tc_peak, "peak_source": peak_src + " (burst bf16)"}


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        gpu_arm(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
