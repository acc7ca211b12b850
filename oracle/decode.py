"""One denoising step of block-wise masked-diffusion decoding, in plain NumPy fp32.

Test infrastructure only (see the package docstring).  Every function states
the passage it follows.  Sources:

* prednext.com "拡散言語モデル (diffusion language model)" explainer, section
  "拡散言語モデルで推論するには": the decoding procedure -- feed [MASK]s,
  adopt the positions whose output passes a threshold, return the rest to
  [MASK], repeat until no [MASK] is left.
* poko-everyday.com Nemotron-TwoTower article, section "技術/ビジネス面": the
  denoising tower attends bidirectionally inside the block and, by
  cross-attention, to the frozen context tower's state.
* dzen.guru Nemotron TwoTower news, "Что нового" / "Как попробовать?": block of
  16, threshold gamma = 0.8 (higher gamma = more quality), the mock-AR mode
  that commits one token per step through the diffusion tower.

Where the pages are silent the readings are fixed here:

* denoiser = pre-norm dense transformer: RMSNorm -> GQA attention -> residual
  -> RMSNorm -> SwiGLU -> residual, L layers, final RMSNorm, untied LM head;
* one softmax per query over [T context keys | S in-block keys], no mask,
  scale 1/sqrt(D); query head h reads kv head h // (Hq/Hkv);
* a learned position table Pos[S,H] is added at the embedding; the [MASK]
  id is V (row V of the embedding); the LM head has V outputs;
* confidence = the largest softmax probability over the V logits
  (temperature 1); argmax ties go to the lowest vocab id;
* commit every masked position with confidence >= gamma; if none qualifies,
  commit the single most confident masked position (lowest position on
  ties); mock-AR commits the leftmost masked position;
* RMSNorm eps = 1e-5, gains from the weights (ones in the synthetic set),
  silu(x) = x / (1 + exp(-x));
* weights and context K/V are bf16 values; every activation is fp32 (the
  default).  `act_bf16=True` instead stores the normalised GEMM inputs,
  q/k/v, the attention output and the SwiGLU product in bf16 the way a bf16
  model would; it exists to measure how far bf16 storage alone moves the
  result (several tenths of a logit after a few layers, because rounding
  flips compound), which is why the fp32 reading is the reference.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

MODE_THRESHOLD = 0
MODE_MOCK_AR = 1
MODE_TOPK = 2     # with k: commit the k most confident masked positions
MODE_STEPS = 3    # with N: the fixed-steps schedule (N denoising steps per block)


def with_param(mode: int, param: int) -> int:
    """A commit mode with its parameter (k or N) in bits 8 and up."""
    return mode | (param << 8)


def steps_schedule_k(block: int, n_steps: int, left: int) -> int:
    """Positions the fixed-steps schedule commits when `left` are masked.

    The schedule starts from `block` masked positions and at its step t
    commits ceil(left_t / (N - t)), so the block fills in exactly N steps
    (N <= block).  The step index is not carried: t is the first step of the
    schedule whose count is at most `left`.
    """
    rem, t = block, 0
    while rem > left and t < n_steps:
        rem -= -(-rem // (n_steps - t))
        t += 1
    steps_left = n_steps - t
    return left if steps_left <= 0 else -(-left // steps_left)

F32 = np.float32

# Near-tie thresholds: a position whose top-2 logit gap or whose distance from
# gamma is below these is reported rather than compared bit-exactly.
TIE_LOGIT_GAP = 1e-2
TIE_GAMMA_GAP = 1e-3
TIE_CONF_GAP = 1e-3


def round_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 -> nearest bf16 (ties to even) -> fp32, elementwise."""
    a = np.ascontiguousarray(x, dtype=F32)
    bits = a.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    rounded = ((bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    return rounded.astype(np.uint32).view(F32).reshape(a.shape)


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """y = x / sqrt(mean(x^2) + eps) * g over the last axis (reading c1/c14)."""
    x = x.astype(F32, copy=False)
    ms = np.mean(x * x, axis=-1, keepdims=True, dtype=F32)
    return (x / np.sqrt(ms + F32(eps))) * g.astype(F32)


def silu(x: np.ndarray) -> np.ndarray:
    """silu(x) = x / (1 + e^-x)."""
    x = x.astype(F32, copy=False)
    return x / (F32(1.0) + np.exp(-x))


def rope(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Rotary positions for the block's queries or keys (reading: interleaved
    pairs; the pages are silent).  x [S, heads, D] fp32; the pair (2j, 2j+1) of
    every head at position p turns by p * theta^(-2j/D) radians (angle, cosine
    and sine in double, the rotation in fp32).
    """
    D = x.shape[-1]
    freq = float(theta) ** (-2.0 * np.arange(D // 2, dtype=np.float64) / D)
    ang = np.asarray(positions, np.float64)[:, None] * freq[None, :]
    c = np.cos(ang).astype(F32)[:, None, :]
    s = np.sin(ang).astype(F32)[:, None, :]
    x = x.astype(F32, copy=False)
    out = np.empty_like(x)
    out[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
    out[..., 1::2] = x[..., 0::2] * s + x[..., 1::2] * c
    return out


def block_attention(q, k_blk, v_blk, k_ctx, v_ctx):
    """Block attention for one sequence.

    Bidirectional over the block plus cross-attention to the context
    (TwoTower article, "技術/ビジネス面"), as one softmax per query over the
    concatenated keys [context | block].  No mask.

    q      [S, Hq, D]      k_blk, v_blk [S, Hkv, D]
    k_ctx, v_ctx [Hkv, T, D] (T may be 0)
    returns [S, Hq, D] fp32
    """
    S, Hq, D = q.shape
    Hkv = k_blk.shape[1]
    G = Hq // Hkv
    scale = F32(1.0 / np.sqrt(D))
    out = np.empty((S, Hq, D), F32)
    for h in range(Hq):
        kvh = h // G
        keys = np.concatenate([k_ctx[kvh], k_blk[:, kvh, :]], axis=0).astype(F32)
        vals = np.concatenate([v_ctx[kvh], v_blk[:, kvh, :]], axis=0).astype(F32)
        s = (q[:, h, :].astype(F32) @ keys.T) * scale          # [S, T+S]
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True, dtype=F32)
        out[:, h, :] = p @ vals
    return out


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y = x W^T in fp32 for a weight stored [out, in]."""
    return x.astype(F32, copy=False) @ w.astype(F32, copy=False).T


def select_from_logits(logits: np.ndarray):
    """Per row: confidence = max softmax probability, argmax (lowest id on ties).

    The explainer adopts positions by the size of the network's output
    ("出力値の大きさ"); the reading here is the top softmax probability at
    temperature 1: conf = 1 / sum_v exp(l_v - l_max).
    Returns (conf fp32 [R], argmax int32 [R]).
    """
    logits = logits.astype(F32, copy=False)
    arg = np.argmax(logits, axis=1).astype(np.int32)           # first maximum
    m = logits.max(axis=1, keepdims=True)
    s = np.exp(logits - m).sum(axis=1, dtype=F32)
    conf = (F32(1.0) / s).astype(F32)
    return conf, arg


def lm_head_select(h: np.ndarray, w_lm: np.ndarray):
    """logits = h W_lm^T (fp32), then `select_from_logits`.  Returns (conf, arg, logits)."""
    logits = h.astype(F32) @ w_lm.astype(F32).T
    conf, arg = select_from_logits(logits)
    return conf, arg, logits


def top2_gap(logits: np.ndarray) -> np.ndarray:
    """Per row: largest logit minus the second largest (0 on an exact tie)."""
    top2 = -np.partition(-logits, 1, axis=1)[:, :2]
    return (top2[:, 0] - top2[:, 1]).astype(np.float64)


def near_tie_flags(logits: np.ndarray, conf: np.ndarray, gamma: float):
    """Rows whose argmax or threshold decision is fragile under rounding.

    A row is flagged when its top-2 logit gap is below TIE_LOGIT_GAP or its
    confidence lies within TIE_GAMMA_GAP of gamma.  This is a per-row
    statement over every row (masked or not); `near_tie_positions` gives the
    per-position flags that decide which commits may differ.
    """
    return (top2_gap(logits) < TIE_LOGIT_GAP) | (np.abs(conf.astype(np.float64) - gamma) < TIE_GAMMA_GAP)


def near_tie_positions(logits, conf, mask, gamma: float, mode: int, block: int) -> np.ndarray:
    """Masked positions whose commit outcome is fragile under rounding (the
    parity bar's near-ties).  Returns bool [B, S]; committed positions are
    never flagged (the commit rule cannot change them).

    A masked position i of sequence b is flagged when
      * its top-2 logit gap is below TIE_LOGIT_GAP (its argmax id may differ), in
        every mode;
      * threshold mode: its confidence is within TIE_GAMMA_GAP of gamma (the
        ">= gamma" decision may differ);
      * threshold mode, fallback (no masked confidence reaches gamma): the two
        largest masked confidences are closer than TIE_CONF_GAP, and conf_i is
        within TIE_CONF_GAP of the largest (the choice of the single most
        confident position may differ);
      * top-k and fixed-steps modes, with k positions to commit out of r > k
        masked: the k-th and (k+1)-th largest masked confidences are closer than
        TIE_CONF_GAP, and conf_i is within TIE_CONF_GAP of either (the cut may
        differ).
    Mock-AR commits the leftmost masked position whatever the confidences, so
    only the logit-gap flag applies there.
    """
    conf = np.asarray(conf, np.float64).reshape(-1, block)
    mask = np.asarray(mask, np.uint32)
    B, S = conf.shape
    gap = top2_gap(np.asarray(logits)).reshape(B, S)
    base, param = mode & 0xFF, mode >> 8
    flags = np.zeros((B, S), bool)
    for b in range(B):
        masked = [i for i in range(S) if (int(mask[b]) >> i) & 1]
        for i in masked:
            if gap[b, i] < TIE_LOGIT_GAP:
                flags[b, i] = True
        if not masked:
            continue
        c = sorted((conf[b, i] for i in masked), reverse=True)
        if base == MODE_THRESHOLD:
            for i in masked:
                if abs(conf[b, i] - gamma) < TIE_GAMMA_GAP:
                    flags[b, i] = True
            fallback = not any(F32(conf[b, i]) >= F32(gamma) for i in masked)
            if fallback and len(c) > 1 and c[0] - c[1] < TIE_CONF_GAP:
                for i in masked:
                    if c[0] - conf[b, i] < TIE_CONF_GAP:
                        flags[b, i] = True
        elif base in (MODE_TOPK, MODE_STEPS):
            k = param if base == MODE_TOPK else steps_schedule_k(S, param, len(masked))
            if 0 < k < len(c) and c[k - 1] - c[k] < TIE_CONF_GAP:
                for i in masked:
                    if min(abs(conf[b, i] - c[k - 1]), abs(conf[b, i] - c[k])) < TIE_CONF_GAP:
                        flags[b, i] = True
    return flags


def commit(conf, arg, tokens, mask, gamma: float, mode: int, block: int):
    """Commit rule for one step, per sequence (explainer steps 3-4; mock-AR from
    the TwoTower news page).

    Threshold: every masked position with conf >= gamma, else the most
    confident one.  Mock-AR: the leftmost masked position.  Top-k (the
    explainer's alternative of forcibly adopting the top few): the k most
    confident masked positions.  Fixed steps: top-k with k from
    `steps_schedule_k`.  Confidence ties go to the lower position.

    conf, arg  [B, S]       tokens [B, S] int32 (updated copy returned)
    mask       [B] uint32, bit i set = position i still [MASK]
    Returns (tokens, mask, n_committed [B] int32, fallback [B] bool) where
    fallback marks sequences where no position reached gamma.
    """
    tokens = np.array(tokens, dtype=np.int32, copy=True)
    mask = np.array(mask, dtype=np.uint32, copy=True)
    B = tokens.shape[0]
    n = np.zeros(B, np.int32)
    fallback = np.zeros(B, bool)
    g = F32(gamma)
    for b in range(B):
        masked = [i for i in range(block) if (int(mask[b]) >> i) & 1]
        if not masked:
            continue
        base, param = mode & 0xFF, mode >> 8
        if base in (MODE_TOPK, MODE_STEPS):
            k = param if base == MODE_TOPK else steps_schedule_k(block, param, len(masked))
            ranked = sorted(masked, key=lambda i: (-float(F32(conf[b, i])), i))
            chosen = sorted(ranked[:k])
        elif mode == MODE_MOCK_AR:
            chosen = [masked[0]]
        else:
            chosen = [i for i in masked if F32(conf[b, i]) >= g]
            if not chosen:
                fallback[b] = True
                best = masked[0]
                for i in masked[1:]:
                    if F32(conf[b, i]) > F32(conf[b, best]):
                        best = i
                chosen = [best]
        bits = int(mask[b])
        for i in chosen:
            tokens[b, i] = arg[b, i]
            bits &= ~(1 << i)
        mask[b] = bits
        n[b] = len(chosen)
    return tokens, mask, n, fallback


@dataclass
class OracleModel:
    """Weights as fp32 arrays holding bf16-rounded values.

    w: dict with embed [V+1,H], pos [S,H], per layer wq/wk/wv/wo/wg/wu/wd
       ([out,in]) and g_attn/g_mlp [H], g_final [H], lm_head [V,H].
    k_ctx, v_ctx: [L][B][Hkv][T][D] (only the first `ctx_len` positions are read).
    """

    cfg: object
    w: dict
    k_ctx: np.ndarray
    v_ctx: np.ndarray
    ctx_len: int

    @staticmethod
    def from_bits(cfg, w_bits: dict, k_bits, v_bits, widen):
        w = {k: widen(v) for k, v in w_bits.items()}
        return OracleModel(cfg, w, widen(k_bits), widen(v_bits), int(k_bits.shape[3]))


@dataclass
class StepResult:
    tokens: np.ndarray
    mask: np.ndarray
    n_committed: np.ndarray
    conf: np.ndarray             # [B,S]
    arg: np.ndarray              # [B,S]
    logits: np.ndarray           # [B*S, V]
    near_tie: np.ndarray         # [B,S] bool: masked positions whose commit may differ (near_tie_positions)
    logit_tie: np.ndarray        # [B,S] bool: every row whose top-2 logit gap is below TIE_LOGIT_GAP
    fallback: np.ndarray         # [B] bool
    attn_out: list = field(default_factory=list)   # per layer [B*S, Hq*D]
    hidden_final: np.ndarray | None = None          # [B*S, H] final-norm output


def denoise_step(model: OracleModel, tokens, mask, gamma: float, mode: int = MODE_THRESHOLD,
                 act_bf16: bool = False, keep_intermediates: bool = False) -> StepResult:
    """One reverse-process application over the block, then the commit rule.

    Explainer step 2 ("逆過程ネットワークに入力する") with the TwoTower denoiser
    reading; steps 3-4 via `commit`.
    """
    cfg, w = model.cfg, model.w
    B, S, H = cfg.batch, cfg.block, cfg.hidden
    Hq, Hkv, D, V = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.vocab
    T = model.ctx_len
    st = round_bf16 if act_bf16 else (lambda a: a.astype(F32, copy=False))
    tokens = np.asarray(tokens, np.int32)
    mask = np.asarray(mask, np.uint32)

    # embedding: [MASK] positions read row V (reading c3/c4)
    ids = np.array([[V if (int(mask[b]) >> i) & 1 else int(tokens[b, i]) for i in range(S)]
                    for b in range(B)], np.int64)
    x = (w["embed"][ids] + w["pos"][None, :, :]).reshape(B * S, H).astype(F32)

    attn_outs = []
    for l in range(cfg.n_layers):
        y = st(rmsnorm(x, w[f"g_attn{l}"], cfg.rms_eps))
        q = (y @ w[f"wq{l}"].T).reshape(B, S, Hq, D)
        k = (y @ w[f"wk{l}"].T).reshape(B, S, Hkv, D)
        if getattr(cfg, "rope_theta", 0.0) > 0:
            # block position i sits at T + i, right after the T context positions
            pos = T + np.arange(S)
            q = np.stack([rope(q[b], pos, cfg.rope_theta) for b in range(B)])
            k = np.stack([rope(k[b], pos, cfg.rope_theta) for b in range(B)])
        q, k = st(q), st(k)
        v = st(y @ w[f"wv{l}"].T).reshape(B, S, Hkv, D)
        o = np.empty((B, S, Hq, D), F32)
        for b in range(B):
            o[b] = block_attention(q[b], k[b], v[b], model.k_ctx[l, b, :, :T], model.v_ctx[l, b, :, :T])
        o = st(o.reshape(B * S, Hq * D))
        if keep_intermediates:
            attn_outs.append(o.copy())
        x = x + o @ w[f"wo{l}"].T
        y = st(rmsnorm(x, w[f"g_mlp{l}"], cfg.rms_eps))
        hmid = st(silu(y @ w[f"wg{l}"].T) * (y @ w[f"wu{l}"].T))
        x = x + hmid @ w[f"wd{l}"].T

    hf = st(rmsnorm(x, w["g_final"], cfg.rms_eps))
    conf, arg, logits = lm_head_select(hf, w["lm_head"])
    conf = conf.reshape(B, S)
    arg = arg.reshape(B, S)
    new_tok, new_mask, n, fallback = commit(conf, arg, tokens, mask, gamma, mode, S)
    tie = near_tie_positions(logits, conf, mask, gamma, mode, S)
    logit_tie = (top2_gap(logits) < TIE_LOGIT_GAP).reshape(B, S)
    return StepResult(new_tok, new_mask, n, conf, arg, logits if keep_intermediates else None,
                      tie, logit_tie, fallback, attn_outs, hf if keep_intermediates else None)


def tower_causal_attention(q, k, v):
    """Causal self-attention inside one committed block: position i attends to
    positions j <= i, one softmax per (query position, head), scale 1/sqrt(D).

    q, k, v [S, heads, D] fp32 -> [S, heads, D] fp32.
    """
    S, Hc, D = q.shape
    scale = F32(1.0 / np.sqrt(D))
    out = np.empty((S, Hc, D), F32)
    for h in range(Hc):
        s = (q[:, h, :] @ k[:, h, :].T) * scale                 # [S, S]
        s = np.where(np.tril(np.ones((S, S), bool)), s, F32(-np.inf))
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True, dtype=F32)
        out[:, h, :] = p @ v[:, h, :]
    return out


def append_block(model: OracleModel, tower: dict, tokens) -> OracleModel:
    """The context tower's encoding of a committed block, appended to the
    context (TwoTower article, "技術/ビジネス面": a frozen causal tower encodes
    the committed tokens and the denoiser cross-attends to its state).  The
    trained tower is out of scope; its stand-in is one causal self-attention
    layer over the committed block followed by the K/V projections:

      e_i = E_ctx[t_i]                      y_i = RMSNorm(e_i) * g
      q_i, k_i, v_i = y_i Wq^T, y_i Wk^T, y_i Wv^T      (Hkv heads of D)
      a_i = causal attention of position i over positions j <= i of the block
      h_i = e_i + a_i Wo^T                  z_i = RMSNorm(h_i) * g2
      for every denoiser layer l: the K rows then the V rows z_i W_kv[l]^T,
      stored in bf16 like the rest of the context at positions [T, T + S).

    Position i of the appended block therefore depends on the committed
    tokens at positions <= i only.  Returns the model with the longer context.

    tower: "ctx_embed" [V, H], "ctx_g" [H], "ctx_wqkv" [3*Hkv*D, H] (q rows,
    then k, then v), "ctx_wo" [H, Hkv*D], "ctx_g2" [H], "ctx_wkv" [L, 2*Hkv*D, H]
    (fp32 holding bf16 values).
    """
    cfg = model.cfg
    B, S, L = cfg.batch, cfg.block, cfg.n_layers
    Hkv, D = cfg.n_kv_heads, cfg.head_dim
    T = model.ctx_len
    ids = np.asarray(tokens, np.int64).reshape(B * S)
    e = tower["ctx_embed"][ids].astype(F32)                                 # [B*S, H]
    y = rmsnorm(e, tower["ctx_g"], cfg.rms_eps)
    qkv = linear(y, tower["ctx_wqkv"]).reshape(B, S, 3, Hkv, D)
    a = np.stack([tower_causal_attention(qkv[b, :, 0], qkv[b, :, 1], qkv[b, :, 2]) for b in range(B)])
    h = e + linear(a.reshape(B * S, Hkv * D), tower["ctx_wo"])
    z = rmsnorm(h, tower["ctx_g2"], cfg.rms_eps)
    k_new = np.empty((L, B, Hkv, S, D), F32)
    v_new = np.empty((L, B, Hkv, S, D), F32)
    for l in range(L):
        kv = round_bf16(z @ tower["ctx_wkv"][l].astype(F32).T)         # [B*S, 2*Hkv*D]
        k_new[l] = kv[:, :Hkv * D].reshape(B, S, Hkv, D).transpose(0, 2, 1, 3)
        v_new[l] = kv[:, Hkv * D:].reshape(B, S, Hkv, D).transpose(0, 2, 1, 3)
    k = np.concatenate([model.k_ctx[:, :, :, :T], k_new], axis=3)
    v = np.concatenate([model.v_ctx[:, :, :, :T], v_new], axis=3)
    return OracleModel(cfg, model.w, k, v, T + S)


def decode_block(model: OracleModel, gamma: float, mode: int = MODE_THRESHOLD,
                 max_steps: int | None = None, act_bf16: bool = False):
    """Fill one block: start all-[MASK], step until no position is masked
    (explainer step 5).  Returns (tokens [B,S], steps, per-step commit counts)."""
    cfg = model.cfg
    S = cfg.block
    max_steps = 4 * S if max_steps is None else max_steps
    tokens = np.full((cfg.batch, S), cfg.vocab, np.int32)
    mask = np.full(cfg.batch, (1 << S) - 1, np.uint32)
    history = []
    steps = 0
    while int(mask.max()) != 0:
        if steps >= max_steps:
            raise RuntimeError("step limit reached before the block filled")
        r = denoise_step(model, tokens, mask, gamma, mode, act_bf16)
        tokens, mask = r.tokens, r.mask
        history.append(r.n_committed)
        steps += 1
    return tokens, steps, history
