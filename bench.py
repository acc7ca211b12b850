"""Benchmark: committed tokens/s of block-wise masked-diffusion decoding on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config large|small|tiny] [--gamma 0.8] [--mode threshold|mock_ar|topk:K|steps:N]

The default workload is the large decode configuration (batch 32, context
32768, block 16, hidden 4096, 32 q / 8 kv heads x 128, 8 layers, SwiGLU 14336,
vocab 131072) at gamma 0.8, the largest that fits one GPU.  One step = one
pass of the whole hot path over one batch: the decode of consecutive
16-position blocks for every sequence of the batch (2 blocks for the large
workload, 8 for the small and tiny ones; each block runs denoising steps until
no position is masked; after each block the context grows by 16 fresh K/V
positions, standing in for the frozen context tower encoding the committed
block).  Inputs are synthetic and seeded (random weights; no datasets or
trained checkpoints exist here).

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

BLOCKS_PER_STEP = {"tiny": 8, "small": 8, "large": 2}
# CPU oracle sample: stop after the denoising step at which this much oracle time has passed
ORACLE_SAMPLE_S = 20.0
METRIC = "committed tokens/sec on 1 B300 (block 16, γ=0.8); block-attn HBM GB/s vs peak"
UNIT = "tokens/s"


def oracle_threads() -> int:
    """Threads the oracle's arithmetic runs on: the size of NumPy's BLAS
    thread pool (its matrix products).  Asked of threadpoolctl where it is
    installed, else of the OpenBLAS that NumPy bundles; failing both, the
    thread count OpenBLAS takes by default (its environment variables, else
    the CPUs this process may use)."""
    try:
        from threadpoolctl import threadpool_info
        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:  # not installed, or the BLAS not introspectable
        pass
    import ctypes
    import glob
    libs = os.path.join(os.path.dirname(os.path.dirname(np.__file__)), "numpy.libs")
    for path in sorted(glob.glob(os.path.join(libs, "*openblas*.so*"))):
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for sym in ("scipy_openblas_get_num_threads64_", "openblas_get_num_threads64_", "openblas_get_num_threads"):
            f = getattr(lib, sym, None)
            if f is not None:
                f.restype = ctypes.c_int
                return int(f())
    cpus = len(os.sched_getaffinity(0))
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        v = os.environ.get(var, "")
        if v.isdigit() and int(v) > 0:
            return min(int(v), cpus)
    return cpus


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
    ap.add_argument("--config", default="large", choices=["tiny", "small", "large"])
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
    ap.add_argument("--no-compact", action="store_true",
                    help="run every sequence's rows in every denoising step (default: only the sequences that "
                         "still have a masked position)")
    ap.add_argument("--no-micro", action="store_true", help="skip the attention / LM-head microbenchmarks")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline and near-tie sample")
    ap.add_argument("--no-small", action="store_true",
                    help="skip the extra short run of the small workload (reported beside the large one)")
    return ap.parse_args(argv)


def workload_desc(cfg, gamma, mode, tower=False):
    return (f"{cfg.name} decode: batch {cfg.batch}, context {cfg.ctx_len} (+16 per block, "
            f"{BLOCKS_PER_STEP[cfg.name]} consecutive blocks), block {cfg.block}, hidden {cfg.hidden}, "
            f"{cfg.n_q_heads} q / {cfg.n_kv_heads} kv heads x d{cfg.head_dim}, {cfg.n_layers} layers, "
            f"SwiGLU {cfg.mlp}, vocab {cfg.vocab}, gamma {gamma}, {mode}"
            + (f", RoPE theta {cfg.rope_theta:g}" if cfg.rope_theta > 0 else "")
            + (", context grown on the device by the context tower" if tower else ""))


def bench_cfg(name, rope_theta=0.0):
    cfg = synth.CONFIGS[name]
    return cfg.replace(max_ctx=cfg.ctx_len + BLOCKS_PER_STEP[name] * cfg.block, rope_theta=rope_theta)


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
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,clocks.mem")

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
        sm, mx, reasons, mem, power = [], 0.0, set(), [], []
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
            for lst, k in ((power, 3), (mem, 9)):
                try:
                    lst.append(float(f[k]))
                except (ValueError, IndexError):
                    pass
        if not sm:
            return None
        out = {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}
        if mem:
            out["mem_mhz"] = float(np.median(mem))
        if power:
            out["power_w"] = float(np.median(power))
        return out


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

def oracle_model_seq0(cfg, w, k, v, T0):
    """The oracle's model of sequence 0 of a workload (batch 1), from the same
    inputs the CUDA path gets: weights as np.uint16 bf16 bits or bf16 torch
    tensors, context K/V [L][B][Hkv][T][D] likewise (only sequence 0 is read)."""
    import oracle

    def f32(t):
        if isinstance(t, np.ndarray):
            return synth.bf16_bits_to_f32(t)
        return t.float().cpu().numpy()
    wf = {n: f32(t) for n, t in w.items()}
    ks = f32(k[:, :1]) if isinstance(k, np.ndarray) else k[:, :1].float().cpu().numpy()
    vs = f32(v[:, :1]) if isinstance(v, np.ndarray) else v[:, :1].float().cpu().numpy()
    return oracle.OracleModel(cfg.replace(batch=1), wf, ks, vs, T0)


def reference_inputs(cfg, seed=0):
    """Inputs of one sequence of the workload for the reference arm: NumPy draws
    for the small and tiny workloads, torch draws (on the GPU when there is
    one) for the large one, whose weights NumPy would take minutes to draw."""
    c = cfg.replace(batch=1)
    if cfg.name != "large":
        kb, vb = synth.make_context_kv(c, seed)
        return synth.make_weights(c, seed), kb, vb
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    w = synth.make_weights_torch(c, seed, dev)
    k, v = synth.make_context_kv_torch(c, 1, dev)
    return w, k, v


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle as it stands, on the host cores.  Each
    step is one oracle denoising step of one sequence of the workload, walking
    the decode of a block (a fresh all-[MASK] block once one fills), so the
    rate is the oracle's committed tokens per second of its own decoding."""
    cfg = bench_cfg(args.config, args.rope_theta)
    if rank != 0:
        return
    import oracle
    w, k, v = reference_inputs(cfg)
    model = oracle_model_seq0(cfg, w, k, v, cfg.ctx_len)
    del w, k, v
    mode = mode_code(args.mode)
    S = cfg.block
    state = {"tok": np.full((1, S), cfg.vocab, np.int32), "mask": np.full(1, (1 << S) - 1, np.uint32)}

    def step():
        r = oracle.denoise_step(model, state["tok"], state["mask"], args.gamma, mode)
        state["tok"], state["mask"] = r.tokens, r.mask
        if int(r.mask[0]) == 0:
            state["tok"] = np.full((1, S), cfg.vocab, np.int32)
            state["mask"] = np.full(1, (1 << S) - 1, np.uint32)
        return int(r.n_committed[0])

    for _ in range(args.warmup):
        step()
    committed = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        committed += step()
    dt = time.perf_counter() - t0
    value = committed / dt
    sample = (f"oracle (NumPy fp32, {oracle_threads()} host threads): {args.steps} denoising steps of one sequence "
              f"of the {cfg.name} workload after {args.warmup} untimed ones, walking a block's decode "
              f"({committed} positions committed in {dt:.1f} s); sequences are independent, so the batch's "
              f"rate is the same per-sequence rate (its work scales with the batch)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": workload_desc(cfg, args.gamma, args.mode), "tokens_per_step": committed / args.steps,
                       "parallelism": f"host cores ({oracle_threads()} threads), rank 0 only",
                       "sample": "one sequence of the workload, one denoising step per step"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def oracle_sample(dec, model, cfg, T0, gamma, mode, dev, budget_s=ORACLE_SAMPLE_S):
    """State-synced oracle sample on sequence 0: the CUDA path decodes a block
    of the whole batch one denoising step at a time (dd_denoise_step); before
    each step the oracle runs the same step for sequence 0 from the CUDA
    path's state.  Returns the oracle's rate (CPU baseline) and the near-tie
    counts: masked positions the oracle flags, masked positions compared, and
    positions where the two sides differ outside a flag (0 when parity holds).
    Stops when sequence 0's block is full or after the step at which
    `budget_s` of oracle time has passed."""
    import oracle
    import torch
    S = cfg.block
    dec.set_context_len(T0)
    t = torch.full((cfg.batch, S), cfg.vocab, dtype=torch.int32, device=dev)
    m = torch.full((cfg.batch,), (1 << S) - 1, dtype=torch.int32, device=dev)
    tok = np.full((1, S), cfg.vocab, np.int32)
    mask = np.full(1, (1 << S) - 1, np.uint32)
    spent, committed, steps, flagged, compared, outside = 0.0, 0, 0, 0, 0, 0
    commits = []
    while int(mask[0]) and steps < 4 * S:
        dec.denoise_step(t, m, gamma, mode)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        r = oracle.denoise_step(model, tok, mask, gamma, mode)
        spent += time.perf_counter() - t0
        g_tok = t[:1].cpu().numpy()
        g_mask = m[:1].cpu().numpy().view(np.uint32)
        masked = ((mask[:, None] >> np.arange(S)) & 1).astype(bool)
        diff = (g_tok != r.tokens) | ((((g_mask[:, None] >> np.arange(S)) & 1) != ((r.mask[:, None] >> np.arange(S)) & 1)))
        flagged += int((r.near_tie & masked).sum())
        compared += int(masked.sum())
        outside += int((diff & ~r.near_tie).sum())
        committed += int(r.n_committed[0])
        commits.append(int(r.n_committed[0]))
        steps += 1
        tok, mask = g_tok, g_mask
        if spent >= budget_s:
            break
    return {"value": committed / spent if spent else None, "seconds": spent, "steps": steps,
            "committed": committed, "commits_per_step": commits, "flagged": flagged, "compared": compared,
            "outside_flags": outside}


# ---------------------------------------------------------------- GPU arm

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of a kernel over
# its algorithmic bytes, from one ncu capture of the same kernel (at the same
# workload, or at a smaller case of the same shapes: traffic grows with the
# units processed, so the ratio carries over); the line's `traffic` is this
# ratio times the launch's algorithmic bytes.  Kinds and workloads not
# captured report null.
TRAFFIC = {("small", "gemm_gate_up"): ((47.241e6 + 0.351e6) / 49545216,
                                       "ncu capture of the small workload's gate|up launch"),
           ("large", "attention_context"): ((4303.529e6 + 32.699e6) / (2 * 2 * 32 * 8 * 32768 * 128 + 2 * 512 * 10240),
                                            "ncu capture of k_attn_ctx_stk<4> at the large layer shapes "
                                            "(32 sequences, 1 layer), ratio of DRAM to algorithmic bytes")}


def algorithmic_bytes(cfg, kind, ctx_len, n_act=None):
    """Minimum HBM bytes of one launch of `kind` (weights/KV read once,
    activations in and out at their stored precision) when `n_act` sequences
    are active (all of the batch by default): with active-sequence compaction
    a launch reads the context K/V and activation rows of those only."""
    n_act = cfg.batch if n_act is None else n_act
    R, H, F, V = n_act * cfg.block, cfg.hidden, cfg.mlp, cfg.vocab
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
        return 2 * 2 * n_act * cfg.n_kv_heads * ctx_len * cfg.head_dim + 2 * R * (qkvw + HqD)
    return None


def algorithmic_flops(cfg, kind, n_act=None):
    """2*R*K*N of one launch of a linear layer or the LM head over the rows of
    `n_act` active sequences (all of the batch by default); None for other
    kinds."""
    n_act = cfg.batch if n_act is None else n_act
    R, H, F, V = n_act * cfg.block, cfg.hidden, cfg.mlp, cfg.vocab
    HqD = cfg.n_q_heads * cfg.head_dim
    kn = {"gemm_qkv": (H, cfg.qkv_width), "gemm_o": (HqD, H), "gemm_gate_up": (H, 2 * F), "gemm_down": (F, H),
          "lm_head_select": (H, V)}.get(kind)
    return None if kn is None else 2.0 * R * kn[0] * kn[1]


def mlp_gemm_rates(cfg, prof, hbm_peak, tc_sust, peak_src):
    """The MLP GEMMs (gate|up, down) of the step from the per-kind profile: HBM
    rate of their algorithmic bytes, and tensor rate of their algorithmic
    FLOPs (2*R*K*N over the active rows of each launch) and of the FLOPs the
    tensor cores execute (twice that: the activation operand is a bf16 head
    plus a bf16 remainder), against the sustained bf16 peak (kernels timed
    inside a long step)."""
    out = {}
    for kind in ("gemm_gate_up", "gemm_down"):
        if kind not in prof:
            continue
        ms, n, nbytes, flops = prof[kind][:4]
        sec = ms * 1e-3
        tf = flops / sec / 1e12
        gbs = nbytes / sec / 1e9
        out[kind] = {"us_per_launch": 1e3 * ms / n, "hbm_GBps": gbs, "hbm_frac": gbs / hbm_peak,
                     "tflops_algorithmic": tf, "tflops_executed": 2 * tf, "tensor_peak_tflops": tc_sust,
                     "tensor_frac_algorithmic": tf / tc_sust, "tensor_frac_executed": 2 * tf / tc_sust,
                     "peak_source": peak_src + " (sustained bf16)",
                     "rows_note": "FLOPs and bytes count the active sequences' rows of each launch"}
    return out


def step_roofline(cfg, T0, hbm_peak, ms_per_step, denoise_per_step, peak_src, active_frac=1.0):
    """The whole denoising step against HBM: every weight read once, the context
    K/V of every layer read once (mean context over the step's blocks) for
    the active sequences (`active_frac` of the batch on average: sequences
    whose block is full are not run)."""
    H, F, V, L = cfg.hidden, cfg.mlp, cfg.vocab, cfg.n_layers
    HqD = cfg.n_q_heads * cfg.head_dim
    weights = 2 * (L * (cfg.qkv_width * H + H * HqD + 2 * F * H + H * F) + V * H)
    t_mean = T0 + cfg.block * (BLOCKS_PER_STEP[cfg.name] - 1) / 2
    kv = 2 * 2 * L * cfg.batch * active_frac * cfg.n_kv_heads * t_mean * cfg.head_dim
    ideal_us = (weights + kv) / (hbm_peak * 1e9) * 1e6
    measured_us = 1e3 * ms_per_step / max(denoise_per_step, 1e-9)
    return {"bytes_per_denoising_step": weights + kv, "active_sequence_fraction": active_frac,
            "ideal_us": ideal_us, "measured_us": measured_us,
            "frac": ideal_us / measured_us, "peak_GBps": hbm_peak, "peak_source": peak_src}


def gpu_arm(args, world, rank, local):
    import torch

    from block_wise_masked_dd_b300 import build as libbuild

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    libbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    line = measure_workload(args, bench_cfg(args.config, args.rope_theta), dev, world, rank, local, peaks,
                            args.steps, args.warmup, full=True)
    if rank == 0 and args.config == "large" and not args.no_small:
        # the small workload beside it (short run, no CPU leg): its rate and step roofline
        small = measure_workload(args, bench_cfg("small", args.rope_theta), dev, 1, 0, local, peaks,
                                 steps=10, warmup=3, full=False)
        line["small_decode"] = {k: small[k] for k in ("value", "unit", "ms_per_step", "steps", "warmup", "config",
                                                      "step_roofline", "roofline", "clocks")}
    hbm_peak, tc_peak, _, peak_src = peaks
    if not args.no_micro and rank == 0:
        stream = torch.cuda.current_stream(dev)
        line["attn_microbench"] = attn_micro(dev, stream, hbm_peak, peak_src)
        line["lmhead_microbench"] = lmhead_micro(dev, stream, tc_peak, peak_src)
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure_workload(args, cfg, dev, world, rank, local, peaks, steps, warmup, full):
    """Time `steps` bench steps of workload `cfg` after `warmup` untimed ones;
    with `full` also the end-to-end pass through host buffers, the CPU oracle
    sample and the MLP GEMM rates.  Returns the JSON line's fields."""
    import torch

    from block_wise_masked_dd_b300 import binding as B
    from block_wise_masked_dd_b300.decoder import Decoder, bits_to_tensor, pack_weights

    mode = mode_code(args.mode)
    hbm_peak, tc_peak, tc_sust, peak_src = peaks
    nblk = BLOCKS_PER_STEP[cfg.name]
    T0 = cfg.ctx_len
    # weights: the same replica on every rank; context differs per rank
    if cfg.name == "large":
        w = synth.make_weights_torch(cfg, 0, dev)
        k0, v0 = synth.make_context_kv_torch(cfg, 1 + rank, dev)
    else:
        w = synth.make_weights(cfg, 0)
        kb, vb = synth.make_context_kv(cfg, rank)
        k0, v0 = bits_to_tensor(kb, dev), bits_to_tensor(vb, dev)
    want_cpu = full and not args.no_cpu and rank == 0
    model = oracle_model_seq0(cfg, w, k0, v0, T0) if want_cpu else None
    weights = pack_weights(cfg, w, dev)
    del w
    dec = Decoder(cfg, weights, dev)
    if args.no_compact:
        dec.compact_sequences = False
    if args.fused_reduce:
        dec.fused_reduce = True
    if dec.fused_reduce:
        linear = "split-K reduced in the GEMM by groups of " + ", ".join(
            f"{k} {cs}" for k, (cs, _) in dec.fused_plan().items())
    else:
        linear = "split-K partials reduced by separate kernels"
    dec.set_context_kv(k0, v0, 0)
    del k0, v0
    # appended context K/V per block: device copies and pinned host copies (e2e)
    gen = synth.torch_generator(100 + rank, dev)
    app_shape = (cfg.n_layers, cfg.batch, cfg.n_kv_heads, cfg.block, cfg.head_dim)
    app = [(synth.torch_normal_bf16(app_shape, 1.0, gen, dev), synth.torch_normal_bf16(app_shape, 1.0, gen, dev))
           for _ in range(nblk)]
    app_host = [(k.cpu().pin_memory(), v.cpu().pin_memory()) for k, v in app] if full else None
    tokens = torch.empty((nblk, cfg.batch, cfg.block), dtype=torch.int32, device=dev)
    tokens_host = torch.empty((nblk, cfg.batch, cfg.block), dtype=torch.int32).pin_memory()
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
        for blk in range(nblk):
            if args.context_tower:
                # the committed block goes to the context on the device; the
                # host only reads the committed ids
                _, n = dec.decode_block(args.gamma, mode, tokens=tokens[blk])
                dec.append_block(tokens[blk])
                if host:
                    tokens_host[blk].copy_(tokens[blk], non_blocking=True)
                counters["launches"] += 3 + n * per_step_launches + 3  # + embed, GEMM, reduce-append
            else:
                out = tokens_host[blk] if host else tokens[blk]
                _, n = dec.decode_block(args.gamma, mode, tokens=out)
                k, v = app_host[blk] if host else app[blk]
                dec.set_context_kv(k, v, T0 + blk * cfg.block)
                counters["launches"] += 3 + n * per_step_launches + 1  # block init, params, loop init; length
            counters["denoise_steps"] += n

    # ---------------------------------------------------- timed region
    for _ in range(warmup):
        one_step(False)
    torch.cuda.synchronize(dev)
    barrier(world)
    counters.update(denoise_steps=0, launches=0)
    clocks = ClockSampler(local)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    ev0.record(stream)
    for _ in range(steps):
        one_step(False)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    barrier(world)
    ms = ev0.elapsed_time(ev1)
    timed_denoise = counters["denoise_steps"]
    timed_launches = counters["launches"]
    ms_max = max_over_ranks(ms, world)
    tokens_per_step = cfg.batch * cfg.block * nblk
    total_tokens = sum_over_ranks(tokens_per_step * steps, world)
    value = total_tokens / (ms_max / 1e3)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
            "warmup": warmup, "ms_per_step": ms_max / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": workload_desc(cfg, args.gamma, args.mode, args.context_tower),
                       "tokens_per_step": tokens_per_step, "parallelism": f"dp{world} (independent batches)",
                       "denoise_steps_per_block": timed_denoise / (steps * nblk),
                       "linear_layers": linear,
                       "sequences_per_step": ("only those with a masked position (active-sequence compaction)"
                                              if dec.compact_sequences and not dec.fused_reduce else "all"),
                       "l2": "inputs larger than L2 (weights + context K/V per denoising step exceed 126 MB)"},
            "gpu_launches": timed_launches, "clocks": clk}

    # ---------------------------------------------- end to end (host buffers)
    if full:
        counters.update(denoise_steps=0, launches=0)
        torch.cuda.synchronize(dev)
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(steps):
            one_step(True)
        torch.cuda.synchronize(dev)
        e2e_s = max_over_ranks(time.perf_counter() - t0, world)
        h2d = 0 if args.context_tower else nblk * 2 * app_host[0][0].numel() * 2
        line["e2e"] = {"value": total_tokens / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": tokens_per_step * 4}

    # ------------------------------------- per-kernel profile of the step
    # (one block, step by step, CUDA events around every launch; each launch's
    # algorithmic bytes count the sequences active in its step)
    prof = {}
    t_, m_ = (torch.full((cfg.batch, cfg.block), cfg.vocab, dtype=torch.int32, device=dev),
              torch.full((cfg.batch,), (1 << cfg.block) - 1, dtype=torch.int32, device=dev))
    dec.set_context_len(T0)
    nprof = 0
    commits = []  # positions committed per denoising step of the first block (all sequences)
    actives = []  # sequences with a masked position before each step
    compacting = dec.compact_sequences and not dec.fused_reduce

    def mask_words():
        return [int(v) & 0xFFFFFFFF for v in m_.cpu().tolist()]
    words = mask_words()
    left = sum(bin(w_).count("1") for w_ in words)
    while left and nprof < 4 * cfg.block:
        n_act = sum(1 for w_ in words if w_) if compacting else cfg.batch
        actives.append(n_act)
        for kind, msk in B.dd_profile_step(dec.ctx, t_.data_ptr(), m_.data_ptr(), args.gamma, mode,
                                           stream=stream.cuda_stream):
            p = prof.setdefault(kind, [0.0, 0, 0.0, 0.0])
            p[0] += msk
            p[1] += 1
            nb = algorithmic_bytes(cfg, kind, T0, n_act)
            p[2] += nb if nb is not None else float("nan")
            nf = algorithmic_flops(cfg, kind, n_act)
            p[3] += nf if nf is not None else float("nan")
        nprof += 1
        words = mask_words()
        now = sum(bin(w_).count("1") for w_ in words)
        commits.append(left - now)
        left = now
    total_prof = sum(v[0] for v in prof.values())
    kernels = {k: {"launches": v[1], "ms_total": v[0], "share": v[0] / total_prof,
                   "us_per_launch": 1e3 * v[0] / v[1]} for k, v in prof.items()}
    dom = max(prof, key=lambda k: prof[k][0])
    dom_us = 1e3 * prof[dom][0] / prof[dom][1]
    dom_bytes = prof[dom][2] / prof[dom][1]
    roofline = None
    if dom_bytes == dom_bytes:  # not NaN: the kind has an algorithmic byte count
        ach = dom_bytes / (dom_us * 1e-6) / 1e9
        traffic = TRAFFIC.get((cfg.name, dom))
        roofline = {"kernel": dom, "bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s",
                    "frac": ach / hbm_peak, "traffic": traffic[0] * dom_bytes if traffic else None,
                    "traffic_source": traffic[1] if traffic else None, "peak_source": peak_src,
                    "algorithmic_bytes_per_launch": dom_bytes, "us_per_launch": dom_us,
                    "bytes_note": "mean over the profiled block's launches, each counting the sequences active "
                                  "in its step"}
    active_frac = (float(np.mean(actives)) / cfg.batch) if actives else 1.0
    line.update({"roofline": roofline, "kernels": kernels,
                 "commits_per_step": {"first_block": commits, "mean": float(np.mean(commits)) if commits else None,
                                      "active_sequences": actives},
                 "step_roofline": step_roofline(cfg, T0, hbm_peak, ms_max / steps, timed_denoise / max(steps, 1),
                                                peak_src, active_frac)})
    if full:
        line["mlp_gemms"] = mlp_gemm_rates(cfg, prof, hbm_peak, tc_sust, peak_src)

    # --------------------- CPU oracle: baseline rate and near-tie sample
    if model is not None:
        o = oracle_sample(dec, model, cfg, T0, args.gamma, mode, dev)
        del model
        line["cpu_baseline"] = {
            "value": o["value"], "unit": UNIT, "cores": oracle_threads(), "kind": "oracle",
            "sample": (f"oracle (NumPy fp32) on sequence 0 of the {cfg.name} workload at gamma {args.gamma}: "
                       f"{o['steps']} denoising steps of a block from the CUDA path's states, "
                       f"{o['committed']} positions committed in {o['seconds']:.1f} s "
                       f"(commits per step {o['commits_per_step']}); sequences are independent, so the "
                       f"whole batch ({cfg.batch} sequences) would take {cfg.batch}x the time for "
                       f"{cfg.batch}x the tokens, the same rate")}
        line["near_ties"] = {"flagged": o["flagged"], "compared": o["compared"],
                             "frac": o["flagged"] / max(o["compared"], 1), "outside_flags": o["outside_flags"],
                             "sample": (f"masked positions of sequence 0 over the {o['steps']} state-synced steps of "
                                        "the CPU sample; outside_flags counts positions where the CUDA path and "
                                        "the oracle committed differently without a near-tie flag (parity: 0)")}
    dec.close()
    return line


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
