"""Torch-tensor front end of libdd: packs tensors into the C-ABI's pointer
structs and streams.  PyTorch supplies device memory and streams only; every
step of decoding runs in libdd's kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B

MODE_THRESHOLD = B.DD_MODE_THRESHOLD
MODE_MOCK_AR = B.DD_MODE_MOCK_AR
MODE_TOPK = B.DD_MODE_TOPK
MODE_STEPS = B.DD_MODE_STEPS
mode_param = B.DD_MODE_PARAM


def _stream(stream=None) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def config_struct(cfg) -> B.dd_config:
    """dd_config from any object with the synthetic Config field names."""
    return B.dd_config(cfg.batch, cfg.block, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                       cfg.n_layers, cfg.mlp, cfg.vocab, cfg.max_ctx, float(cfg.rms_eps),
                       float(getattr(cfg, "rope_theta", 0.0)))


def bits_to_tensor(bits: np.ndarray, device) -> torch.Tensor:
    """bf16 bit patterns (np.uint16) -> torch.bfloat16 tensor on `device`."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


def pack_weights(cfg, w_bits: dict, device) -> dict:
    """Stack per-layer bf16 weights (np.uint16 bit patterns or bf16 tensors)
    into the layout dd_weights expects."""
    L = cfg.n_layers

    def t(name):
        v = w_bits[name]
        return v if isinstance(v, torch.Tensor) else bits_to_tensor(v, "cpu")
    out = {
        "embed": t("embed"),
        "pos": t("pos"),
        "wqkv": torch.stack([torch.cat([t(f"wq{l}"), t(f"wk{l}"), t(f"wv{l}")], 0) for l in range(L)]),
        "wo": torch.stack([t(f"wo{l}") for l in range(L)]),
        "wgu": torch.stack([torch.cat([t(f"wg{l}"), t(f"wu{l}")], 0) for l in range(L)]),
        "wd": torch.stack([t(f"wd{l}") for l in range(L)]),
        "g_attn": torch.stack([t(f"g_attn{l}") for l in range(L)]),
        "g_mlp": torch.stack([t(f"g_mlp{l}") for l in range(L)]),
        "g_final": t("g_final"),
        "lm_head": t("lm_head"),
    }
    return {k: v.contiguous().to(device) for k, v in out.items()}


def weights_struct(w: dict) -> B.dd_weights:
    return B.dd_weights(*[_ptr(w[n]) for n in ("embed", "pos", "wqkv", "wo", "wgu", "wd", "g_attn", "g_mlp",
                                                "g_final", "lm_head")])


class Decoder:
    """One libdd context over a torch-allocated workspace."""

    def __init__(self, cfg, weights: dict, device="cuda"):
        self.cfg = cfg
        self.device = torch.device(device)
        self.cstruct = config_struct(cfg)
        nbytes = B.dd_workspace_size(self.cstruct)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        self.weights = weights
        with torch.cuda.device(self.device):
            self.ctx = B.dd_create(self.cstruct, _ptr(self.workspace), nbytes)
            B.dd_init_weights(self.ctx, weights_struct(weights))

    def set_weights(self, weights: dict):
        """Point the context at another set of packed weights (kept alive here)."""
        with torch.cuda.device(self.device):
            B.dd_init_weights(self.ctx, weights_struct(weights))
        self.weights = weights

    def close(self):
        if getattr(self, "ctx", None):
            B.dd_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_context_kv(self, k: torch.Tensor, v: torch.Tensor, t0: int = 0, stream=None):
        """k, v: bf16 [L][B][Hkv][n][D] (device or host); positions [t0, t0+n)."""
        n = int(k.shape[3]) if k is not None else 0
        B.dd_set_context_kv(self.ctx, _ptr(k), _ptr(v), t0, n, _stream(stream))

    def set_context_len(self, n: int, stream=None):
        B.dd_set_context_kv(self.ctx, 0, 0, n, 0, _stream(stream))

    def denoise_step(self, tokens: torch.Tensor, mask: torch.Tensor, gamma: float, mode: int = MODE_THRESHOLD,
                     n_committed: torch.Tensor | None = None, stream=None):
        B.dd_denoise_step(self.ctx, _ptr(tokens), _ptr(mask), gamma, mode, _ptr(n_committed), _stream(stream))

    def decode_block(self, gamma: float, mode: int = MODE_THRESHOLD, max_steps: int = 0,
                     tokens: torch.Tensor | None = None, stream=None):
        if tokens is None:
            tokens = torch.empty((self.cfg.batch, self.cfg.block), dtype=torch.int32, device=self.device)
        steps = B.dd_decode_block(self.ctx, _ptr(tokens), gamma, mode, max_steps, _stream(stream))
        return tokens, steps

    def set_context_tower(self, tower: dict):
        """Register the synthetic context tower: "ctx_embed" [V][H], "ctx_g" [H],
        "ctx_wqkv" [3*Hkv*D][H], "ctx_wo" [H][Hkv*D], "ctx_g2" [H],
        "ctx_wkv" [L][2*Hkv*D][H] (np.uint16 bf16 bits or bf16 tensors; kept
        alive here)."""
        names = ("ctx_embed", "ctx_g", "ctx_wqkv", "ctx_wo", "ctx_g2", "ctx_wkv")

        def t(name):
            v = tower[name]
            return (v if isinstance(v, torch.Tensor) else bits_to_tensor(v, "cpu")).contiguous().to(self.device)
        self.tower = {n: t(n) for n in names}
        B.dd_set_context_tower(self.ctx, *[_ptr(self.tower[n]) for n in names])

    def append_block(self, tokens: torch.Tensor, stream=None):
        """Encode the committed block `tokens` [B][S] (device int32) with the
        context tower and append its K/V to the context."""
        B.dd_append_block(self.ctx, _ptr(tokens), _stream(stream))

    def device_status(self, stream=None):
        """Raise DDError if a kernel of this context recorded an expired bounded wait."""
        B.dd_device_status(self.ctx, _stream(stream))

    @property
    def compact_sequences(self) -> bool:
        """Each step runs only the rows of sequences that still have a masked
        position (default True); probe activations are then in compacted row
        order (see `active_rows`)."""
        return bool(B.dd_get_option(self.ctx, B.DD_OPT_COMPACT_SEQUENCES))

    @compact_sequences.setter
    def compact_sequences(self, on: bool):
        B.dd_set_option(self.ctx, B.DD_OPT_COMPACT_SEQUENCES, 1 if on else 0)

    @property
    def fused_reduce(self) -> bool:
        """Linear layers reduce their K splits inside the GEMM (groups of
        CTAs exchanging partials through L2); False: separate reduce kernels."""
        return bool(B.dd_get_option(self.ctx, B.DD_OPT_FUSED_REDUCE))

    @fused_reduce.setter
    def fused_reduce(self, on: bool):
        B.dd_set_option(self.ctx, B.DD_OPT_FUSED_REDUCE, 1 if on else 0)

    def fused_plan(self) -> dict:
        """{layer: (K splits, grid)} of the fused linear layers (zeros when unavailable)."""
        return {k: (B.dd_get_option(self.ctx, B.DD_OPT_FUSED_SPLITS[k]), B.dd_get_option(self.ctx, B.DD_OPT_FUSED_GRID[k]))
                for k in B.DD_OPT_FUSED_SPLITS}

    def probe_step(self, tokens, mask, gamma, mode=MODE_THRESHOLD, logits=True, stream=None):
        """One step with every probe output; returns a dict of tensors."""
        cfg = self.cfg
        R = cfg.batch * cfg.block
        dev = self.device
        # activations come back as bf16 heads (rows [0,R)) and remainders (rows [R,2R))
        out = {
            "attn_out": torch.empty((cfg.n_layers, 2 * R, cfg.n_q_heads * cfg.head_dim), dtype=torch.bfloat16,
                                    device=dev),
            "hidden": torch.empty((2 * R, cfg.hidden), dtype=torch.bfloat16, device=dev),
            "logits": torch.empty((R, cfg.vocab), dtype=torch.float32, device=dev) if logits else None,
            "conf": torch.empty(R, dtype=torch.float32, device=dev),
            "arg": torch.empty(R, dtype=torch.int32, device=dev),
            "n_committed": torch.empty(cfg.batch, dtype=torch.int32, device=dev),
        }
        p = B.dd_probe(_ptr(out["attn_out"]), _ptr(out["hidden"]), _ptr(out["logits"]), _ptr(out["conf"]),
                       _ptr(out["arg"]))
        B.dd_denoise_step_probe(self.ctx, _ptr(tokens), _ptr(mask), gamma, mode, _ptr(out["n_committed"]), p,
                                _stream(stream))
        return out


def active_rows(mask, block: int, compacted: bool):
    """Original rows (b*S + i) in the order a probe reports them: with
    active-sequence compaction, the rows of the sequences whose mask word is
    non-zero, in sequence order; otherwise every row."""
    m = np.asarray(mask).astype(np.uint32).reshape(-1)
    seqs = np.nonzero(m)[0] if compacted else np.arange(m.size)
    return (seqs[:, None] * block + np.arange(block)[None, :]).reshape(-1)


def join_split(t: torch.Tensor) -> torch.Tensor:
    """fp32 value of a head/remainder bf16 tensor whose second-to-last axis
    holds heads in its first half and remainders in its second half."""
    n = t.shape[-2] // 2
    return t[..., :n, :].float() + t[..., n:, :].float()


# ------------------------------------------------------------- single kernels

def workspace_status(ws: torch.Tensor) -> int:
    """The status word a single-kernel call leaves in the first 4 bytes of its
    workspace: 0, or non-zero if a bounded wait inside a kernel expired."""
    torch.cuda.synchronize(ws.device)
    return int(ws[:4].view(torch.int32).item())


class BlockAttention:
    """dd_block_attention with a persistent workspace (for repeated launches)."""

    def __init__(self, batch, block, n_q_heads, n_kv_heads, head_dim, ctx_len, ctx_stride, device="cuda"):
        self.p = B.dd_attn_problem(batch, block, n_q_heads, n_kv_heads, head_dim, ctx_len, ctx_stride,
                                   0, 0, 0, 0, 0, 0)
        n = B.dd_block_attention_workspace_size(self.p)
        self.workspace = torch.empty(n, dtype=torch.uint8, device=device)
        self.p.workspace = _ptr(self.workspace)
        self.p.workspace_bytes = n

    def __call__(self, qkv, k_ctx, v_ctx, out, stream=None):
        self.p.qkv, self.p.k_ctx, self.p.v_ctx, self.p.out = _ptr(qkv), _ptr(k_ctx), _ptr(v_ctx), _ptr(out)
        B.dd_block_attention(self.p, _stream(stream))
        return out

    def status(self) -> int:
        """The last call's status word (0, or non-zero if a bounded wait expired); synchronises."""
        return workspace_status(self.workspace)


def block_attention(qkv, k_ctx, v_ctx, ctx_len, batch, block, n_q_heads, n_kv_heads, head_dim, stream=None):
    """qkv bf16 [B*S, (Hq+2Hkv)*D]; k_ctx/v_ctx bf16 [B, Hkv, stride, D] -> out bf16 [B*S, Hq*D]."""
    op = BlockAttention(batch, block, n_q_heads, n_kv_heads, head_dim, ctx_len, int(k_ctx.shape[2]), qkv.device)
    out = torch.empty((batch * block, n_q_heads * head_dim), dtype=torch.bfloat16, device=qkv.device)
    return op(qkv, k_ctx, v_ctx, out, stream)


class LmHeadSelect:
    def __init__(self, rows, hidden, vocab, device="cuda"):
        self.rows, self.hidden, self.vocab = rows, hidden, vocab
        n = B.dd_lmhead_select_workspace_size(rows, hidden, vocab)
        self.workspace = torch.empty(n, dtype=torch.uint8, device=device)

    def __call__(self, x, w, conf, arg, stream=None):
        B.dd_lmhead_select(self.rows, self.hidden, self.vocab, _ptr(x), _ptr(w), _ptr(conf), _ptr(arg),
                           _ptr(self.workspace), self.workspace.numel(), _stream(stream))
        return conf, arg

    def status(self) -> int:
        """The last call's status word (0, or non-zero if a bounded wait expired); synchronises."""
        return workspace_status(self.workspace)


def lmhead_select(x, w, stream=None):
    """x bf16 [rows, H], w bf16 [V, H] -> (conf fp32 [rows], arg int32 [rows])."""
    rows, hidden = x.shape
    vocab = w.shape[0]
    op = LmHeadSelect(rows, hidden, vocab, x.device)
    conf = torch.empty(rows, dtype=torch.float32, device=x.device)
    arg = torch.empty(rows, dtype=torch.int32, device=x.device)
    return op(x, w, conf, arg, stream)


def gemm(x, w, stream=None):
    """y = x w^T through the linear-layer tensor-core kernel; x bf16 [rows,k], w bf16 [n,k] -> fp32 [rows,n]."""
    rows, k = x.shape
    n = w.shape[0]
    nb = B.dd_gemm_workspace_size(rows, n, k)
    ws = torch.empty(nb, dtype=torch.uint8, device=x.device)
    y = torch.empty((rows, n), dtype=torch.float32, device=x.device)
    B.dd_gemm(rows, n, k, _ptr(x), _ptr(w), _ptr(y), _ptr(ws), nb, _stream(stream))
    return y


def commit(conf, arg, tokens, mask, gamma, mode=MODE_THRESHOLD, stream=None):
    """The commit rule alone, in place on tokens/mask; returns (n_committed, remaining)."""
    batch, block = tokens.shape
    n = torch.empty(batch, dtype=torch.int32, device=tokens.device)
    rem = torch.empty(1, dtype=torch.int32, device=tokens.device)
    B.dd_commit(batch, block, _ptr(conf), _ptr(arg), _ptr(tokens), _ptr(mask), gamma, mode, _ptr(n), _ptr(rem),
                _stream(stream))
    return n, rem
