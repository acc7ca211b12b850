"""Small, self-contained workloads for profiler captures (ncu).

    python -m block_wise_masked_dd_b300.profile_cases step   [--config small] [--iters N] [--batch B --layers L]
    python -m block_wise_masked_dd_b300.profile_cases attn   [--iters N] [--batch B --ctx T]
                                                    # default B=64, T=8192, 32/8 x 128
    python -m block_wise_masked_dd_b300.profile_cases lmhead [--iters N]   # 1024 x 4096 x 131072
    python -m block_wise_masked_dd_b300.profile_cases gemm   [--rows 128 --n 11264 --k 2048]

Each case builds its inputs (seeded, synthetic), runs one untimed launch, then
`--iters` launches, and prints one line with the mean time from CUDA events.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _time(fn, iters):
    import torch
    fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / max(iters, 1)


def case_step(args):
    import torch

    import synth
    from block_wise_masked_dd_b300.decoder import Decoder, bits_to_tensor, pack_weights
    cfg = synth.CONFIGS[args.config]
    if args.batch:
        cfg = cfg.replace(batch=args.batch)
    if args.layers:
        cfg = cfg.replace(n_layers=args.layers)
    if cfg.name == "large":
        w = synth.make_weights_torch(cfg, 0, "cuda")
        k, v = synth.make_context_kv_torch(cfg, 1, "cuda")
    else:
        w = synth.make_weights(cfg, 0)
        kb, vb = synth.make_context_kv(cfg, 0)
        k, v = bits_to_tensor(kb, "cuda"), bits_to_tensor(vb, "cuda")
    dec = Decoder(cfg, pack_weights(cfg, w, "cuda"), "cuda")
    dec.set_context_kv(k, v, 0)
    del k, v
    tok = torch.full((cfg.batch, cfg.block), cfg.vocab, dtype=torch.int32, device="cuda")
    mask = torch.full((cfg.batch,), (1 << cfg.block) - 1, dtype=torch.int32, device="cuda")

    def step():
        t, m = tok.clone(), mask.clone()
        dec.denoise_step(t, m, args.gamma)

    ms = _time(step, args.iters)
    print(f"step {cfg.name}: {ms * 1e3:.1f} us per denoising step (graph launch, first step of a block)")


def case_attn(args):
    import torch

    import synth
    from block_wise_masked_dd_b300.decoder import BlockAttention
    c = synth.ATTN_MICRO.replace(batch=args.batch or synth.ATTN_MICRO.batch, ctx_len=args.ctx or synth.ATTN_MICRO.ctx_len)
    c = c.replace(max_ctx=c.ctx_len)
    g = synth.torch_generator(7, "cuda")
    qkv = synth.torch_normal_bf16((c.rows, c.qkv_width), 1.0, g, "cuda")
    kc = synth.torch_normal_bf16((c.batch, c.n_kv_heads, c.ctx_len, c.head_dim), 1.0, g, "cuda")
    vc = synth.torch_normal_bf16((c.batch, c.n_kv_heads, c.ctx_len, c.head_dim), 1.0, g, "cuda")
    out = torch.empty((c.rows, c.n_q_heads * c.head_dim), dtype=torch.bfloat16, device="cuda")
    op = BlockAttention(c.batch, c.block, c.n_q_heads, c.n_kv_heads, c.head_dim, c.ctx_len, c.ctx_len, "cuda")
    ms = _time(lambda: op(qkv, kc, vc, out), args.iters)
    nbytes = 4 * c.batch * c.n_kv_heads * c.ctx_len * c.head_dim
    print(f"attn B{c.batch} T{c.ctx_len}: {ms * 1e3:.1f} us per launch, {nbytes / ms / 1e6:.0f} GB/s of context K/V")


def case_lmhead(args):
    import torch

    import synth
    from block_wise_masked_dd_b300.decoder import LmHeadSelect
    rows, H, V = 1024, 4096, 131072
    g = synth.torch_generator(9, "cuda")
    x = synth.torch_normal_bf16((rows, H), 1.0, g, "cuda")
    w = synth.torch_normal_bf16((V, H), synth.LOGIT_STD / np.sqrt(H), g, "cuda")
    conf = torch.empty(rows, dtype=torch.float32, device="cuda")
    arg = torch.empty(rows, dtype=torch.int32, device="cuda")
    op = LmHeadSelect(rows, H, V, "cuda")
    ms = _time(lambda: op(x, w, conf, arg), args.iters)
    print(f"lmhead: {ms * 1e3:.1f} us per launch, {2 * rows * H * V / ms / 1e9:.0f} TFLOP/s")


def case_gemm(args):
    import torch

    import synth
    from block_wise_masked_dd_b300.decoder import gemm
    g = synth.torch_generator(5, "cuda")
    x = synth.torch_normal_bf16((args.rows, args.k), 1.0, g, "cuda")
    w = synth.torch_normal_bf16((args.n, args.k), 0.02, g, "cuda")
    ms = _time(lambda: gemm(x, w), args.iters)
    print(f"gemm {args.rows}x{args.n}x{args.k}: {ms * 1e3:.1f} us per call, "
          f"{2 * args.n * args.k / ms / 1e6:.0f} GB/s of weights")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["step", "attn", "lmhead", "gemm"])
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--config", default="small")
    ap.add_argument("--gamma", type=float, default=0.8)
    ap.add_argument("--batch", type=int, default=0,
                    help="attn: sequences (0: the microbenchmark's 64); step: sequences (0: the workload's)")
    ap.add_argument("--layers", type=int, default=0, help="step: denoiser layers (0: the workload's)")
    ap.add_argument("--ctx", type=int, default=0, help="attn: context length (0: the microbenchmark's 8192)")
    ap.add_argument("--rows", type=int, default=128)
    ap.add_argument("--n", type=int, default=11264)
    ap.add_argument("--k", type=int, default=2048)
    args = ap.parse_args()
    from block_wise_masked_dd_b300 import build as libbuild
    libbuild.build()
    {"step": case_step, "attn": case_attn, "lmhead": case_lmhead, "gemm": case_gemm}[args.case](args)


if __name__ == "__main__":
    main()
