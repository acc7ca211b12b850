"""Seeded synthetic inputs for block-wise masked-diffusion decoding.

This module is the only code shared by the CPU oracle and the CUDA path.
It draws random numbers and rounds them to bf16; it holds none of the
decoding arithmetic (no norm, attention, MLP, softmax or commit rule).

Workload shapes follow the pages' operating point: a block of 16 [MASK]
positions per sequence, confidence threshold 0.8 (Nemotron TwoTower news
page, "Что нового" / "Как попробовать?"), a frozen context tower whose
output is a KV cache (poko-everyday TwoTower article, "技術/ビジネス面").
Trained weights are not available, so every tensor is a seeded normal draw:

* projection / MLP matrices, token and position embeddings: N(0, 0.02)
* LM head: N(0, (8/sqrt(H))^2), so logits have std ~8 after the final RMSNorm
* RMSNorm gains: 1
* context K/V: N(0, 1)

Values are drawn in fp32 and rounded to bf16 (round to nearest, ties to
even).  Small configurations are drawn with NumPy (one SeedSequence
substream per tensor, in a fixed order); the large ones are drawn on the
device with a seeded torch generator, and the oracle gets host copies of
the slices it needs.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np

MODE_THRESHOLD = 0
MODE_MOCK_AR = 1


@dataclass(frozen=True)
class Config:
    """Shape of one decoding problem.

    batch      sequences decoded together (B)
    block      positions per block (S, at most 32)
    hidden     model width (H)
    n_q_heads  query heads (Hq)
    n_kv_heads key/value heads (Hkv), Hq % Hkv == 0
    head_dim   per-head width (D)
    n_layers   denoiser layers (L)
    mlp        SwiGLU width (F)
    vocab      LM-head outputs (V); the embedding has V+1 rows, row V = [MASK]
    ctx_len    context positions present in the KV cache (T)
    max_ctx    capacity of the KV cache (>= ctx_len)
    rms_eps    RMSNorm epsilon
    rope_theta rotary base for the block's queries and keys (0: learned
               in-block positions only)
    """

    name: str
    batch: int
    block: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_layers: int
    mlp: int
    vocab: int
    ctx_len: int
    max_ctx: int
    rms_eps: float = 1e-5
    rope_theta: float = 0.0

    @property
    def rows(self) -> int:
        return self.batch * self.block

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def qkv_width(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    def replace(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


# The five workloads of the decoding study.  TINY is the case the oracle
# finishes in seconds; SMALL a mid-size decode workload; LARGE the largest
# decode workload one GPU holds, the one throughput is quoted on; the two
# microbenchmarks time the block attention and the LM head + select alone.
TINY = Config("tiny", batch=1, block=16, hidden=256, n_q_heads=4, n_kv_heads=4,
              head_dim=64, n_layers=2, mlp=1024, vocab=4096, ctx_len=256, max_ctx=256)
SMALL = Config("small", batch=8, block=16, hidden=2048, n_q_heads=16, n_kv_heads=4,
               head_dim=128, n_layers=4, mlp=5632, vocab=32768, ctx_len=2048,
               max_ctx=2048 + 8 * 16)
ATTN_MICRO = Config("attn_micro", batch=64, block=16, hidden=4096, n_q_heads=32,
                    n_kv_heads=8, head_dim=128, n_layers=1, mlp=0, vocab=0,
                    ctx_len=8192, max_ctx=8192)
LMHEAD_MICRO = Config("lmhead_micro", batch=64, block=16, hidden=4096, n_q_heads=0,
                      n_kv_heads=1, head_dim=128, n_layers=0, mlp=0, vocab=131072,
                      ctx_len=0, max_ctx=0)
LARGE = Config("large", batch=32, block=16, hidden=4096, n_q_heads=32, n_kv_heads=8,
               head_dim=128, n_layers=8, mlp=14336, vocab=131072, ctx_len=32768,
               max_ctx=32768 + 16)

CONFIGS = {c.name: c for c in (TINY, SMALL, ATTN_MICRO, LMHEAD_MICRO, LARGE)}

WEIGHT_STD = 0.02
LOGIT_STD = 8.0


# ---------------------------------------------------------------------------
# bf16 storage helpers (input rounding only)
# ---------------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16, nearest-even; returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to fp32 values (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return to_bf16_bits(x)


# ---------------------------------------------------------------------------
# Weights
# ---------------------------------------------------------------------------

def weight_names(cfg: Config):
    """Tensor names in generation order, with their shapes ([out, in] for matrices)."""
    H, D, F, V = cfg.hidden, cfg.head_dim, cfg.mlp, cfg.vocab
    out = [("embed", (V + 1, H)), ("pos", (cfg.block, H))]
    for l in range(cfg.n_layers):
        out += [(f"wq{l}", (cfg.n_q_heads * D, H)), (f"wk{l}", (cfg.n_kv_heads * D, H)),
                (f"wv{l}", (cfg.n_kv_heads * D, H)), (f"wo{l}", (H, cfg.n_q_heads * D)),
                (f"wg{l}", (F, H)), (f"wu{l}", (F, H)), (f"wd{l}", (H, F))]
    out.append(("lm_head", (V, H)))
    return out


def weight_std(cfg: Config, name: str) -> float:
    return LOGIT_STD / np.sqrt(cfg.hidden) if name == "lm_head" else WEIGHT_STD


def make_weights(cfg: Config, seed: int = 0) -> dict:
    """All weights as bf16 bit patterns (np.uint16), drawn with NumPy.

    Norm gains are all ones and are returned as bf16 bits too
    ("g_attn{l}", "g_mlp{l}", "g_final").
    """
    names = weight_names(cfg)
    streams = np.random.SeedSequence(seed).spawn(len(names))
    w = {}
    for (name, shape), ss in zip(names, streams):
        w[name] = _normal_bf16(np.random.default_rng(ss), shape, weight_std(cfg, name))
    one = to_bf16_bits(np.ones(cfg.hidden, np.float32))
    for l in range(cfg.n_layers):
        w[f"g_attn{l}"] = one.copy()
        w[f"g_mlp{l}"] = one.copy()
    w["g_final"] = one.copy()
    return w


def tower_names(cfg: Config):
    """The synthetic context tower's tensors: its token embedding [V][H], per
    denoiser layer the K rows then the V rows it produces ([L][2*Hkv*D][H]),
    and its causal self-attention layer: q|k|v projection [3*Hkv*D][H] and
    output projection [H][Hkv*D] (drawn after the first two, so their draws
    do not move)."""
    kvd = cfg.n_kv_heads * cfg.head_dim
    return [("ctx_embed", (cfg.vocab, cfg.hidden)),
            ("ctx_wkv", (cfg.n_layers, 2 * kvd, cfg.hidden)),
            ("ctx_wqkv", (3 * kvd, cfg.hidden)),
            ("ctx_wo", (cfg.hidden, kvd))]


def tower_std(cfg: Config, name: str) -> float:
    """Embedding N(0, 0.02); q|k|v and K/V projections N(0, 1/H) so their
    outputs are ~N(0, 1) (like the synthetic context); the attention output
    projection N(0, 0.02^2 / (Hkv*D)), so its contribution is on the scale of
    the embedding it is added to."""
    if name == "ctx_embed":
        return WEIGHT_STD
    if name == "ctx_wo":
        return WEIGHT_STD / np.sqrt(cfg.n_kv_heads * cfg.head_dim)
    return 1.0 / np.sqrt(cfg.hidden)


def make_tower_weights(cfg: Config, seed: int = 0) -> dict:
    """Context-tower weights as bf16 bits (scales in `tower_std`); gains
    "ctx_g" and "ctx_g2" ones."""
    names = tower_names(cfg)
    streams = np.random.SeedSequence([seed, 0x544F57]).spawn(len(names))
    w = {}
    for (name, shape), ss in zip(names, streams):
        w[name] = _normal_bf16(np.random.default_rng(ss), shape, tower_std(cfg, name))
    w["ctx_g"] = to_bf16_bits(np.ones(cfg.hidden, np.float32))
    w["ctx_g2"] = to_bf16_bits(np.ones(cfg.hidden, np.float32))
    return w


def make_context_kv(cfg: Config, seed: int = 0, t0: int = 0, n: int | None = None):
    """Context K and V for positions [t0, t0+n) as bf16 bits, layout [L][B][Hkv][n][D].

    Each (position range) draw uses its own substream keyed by (seed, t0, n),
    so appended blocks are reproducible on their own.
    """
    n = cfg.ctx_len if n is None else n
    shape = (max(cfg.n_layers, 1), cfg.batch, cfg.n_kv_heads, n, cfg.head_dim)
    ss = np.random.SeedSequence([seed, 0x4B56, t0, n])
    sk, sv = ss.spawn(2)
    k = _normal_bf16(np.random.default_rng(sk), shape, 1.0)
    v = _normal_bf16(np.random.default_rng(sv), shape, 1.0)
    return k, v


def make_tokens(cfg: Config, seed: int = 0, masked_frac: float = 1.0):
    """A block state: token ids [B,S] (int32) and mask bitmaps [B] (uint32).

    masked_frac=1 is the start of a block (every position [MASK], ids = V);
    otherwise a seeded subset of positions is already committed with random ids.
    """
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x544F4B]))
    B, S, V = cfg.batch, cfg.block, cfg.vocab
    tok = np.full((B, S), V, np.int32)
    mask = np.zeros(B, np.uint32)
    for b in range(B):
        m = rng.random(S) < masked_frac if masked_frac < 1.0 else np.ones(S, bool)
        if not m.any():
            m[rng.integers(S)] = True
        ids = rng.integers(0, V, size=S, dtype=np.int32)
        tok[b] = np.where(m, V, ids)
        bits = 0
        for i in range(S):
            if m[i]:
                bits |= 1 << i
        mask[b] = bits
    return tok, mask


def make_activations(rows: int, width: int, seed: int = 0, std: float = 1.0) -> np.ndarray:
    """A bf16 activation matrix [rows, width] ~ N(0, std^2) (bits)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x414354, rows, width]))
    return _normal_bf16(rng, (rows, width), std)


# ---------------------------------------------------------------------------
# Device-side draws for the large workloads (torch generator, seeded)
# ---------------------------------------------------------------------------

def torch_normal_bf16(shape, std: float, gen, device, chunk_elems: int = 1 << 28):
    """A bf16 tensor ~ N(0, std^2) drawn on `device` with torch's generator `gen`.

    Drawn in fp32 slices of at most `chunk_elems` elements along the first
    dimension, so a large tensor never needs a full fp32 copy.
    """
    import torch
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1) if len(shape) > 1 else out.view(-1, 1)
    per_row = flat.shape[1]
    rows = max(1, chunk_elems // max(per_row, 1))
    for r0 in range(0, flat.shape[0], rows):
        r1 = min(flat.shape[0], r0 + rows)
        tmp = torch.empty((r1 - r0, per_row), dtype=torch.float32, device=device)
        tmp.normal_(0.0, std, generator=gen)
        flat[r0:r1].copy_(tmp)
    return out


def make_weights_torch(cfg: Config, seed: int, device) -> dict:
    """All weights as bf16 torch tensors drawn on `device` (same names, shapes
    and scales as `make_weights`, different random stream)."""
    import torch
    gen = torch_generator(seed, device)
    w = {name: torch_normal_bf16(shape, weight_std(cfg, name), gen, device) for name, shape in weight_names(cfg)}
    one = torch.ones(cfg.hidden, dtype=torch.bfloat16, device=device)
    for l in range(cfg.n_layers):
        w[f"g_attn{l}"] = one.clone()
        w[f"g_mlp{l}"] = one.clone()
    w["g_final"] = one.clone()
    return w


def make_tower_weights_torch(cfg: Config, seed: int, device) -> dict:
    """Context-tower weights as bf16 torch tensors drawn on `device` (same
    names, shapes and scales as `make_tower_weights`, different stream)."""
    import torch
    gen = torch_generator(seed * 7919 + 0x544F57, device)
    w = {name: torch_normal_bf16(shape, tower_std(cfg, name), gen, device) for name, shape in tower_names(cfg)}
    w["ctx_g"] = torch.ones(cfg.hidden, dtype=torch.bfloat16, device=device)
    w["ctx_g2"] = torch.ones(cfg.hidden, dtype=torch.bfloat16, device=device)
    return w


def make_context_kv_torch(cfg: Config, seed: int, device, t0: int = 0, n: int | None = None):
    """Context K and V on `device`, bf16 [L][B][Hkv][n][D] ~ N(0,1)."""
    n = cfg.ctx_len if n is None else n
    gen = torch_generator(seed * 1000003 + t0 * 7 + n, device)
    shape = (max(cfg.n_layers, 1), cfg.batch, cfg.n_kv_heads, n, cfg.head_dim)
    return torch_normal_bf16(shape, 1.0, gen, device), torch_normal_bf16(shape, 1.0, gen, device)


def torch_generator(seed: int, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g
