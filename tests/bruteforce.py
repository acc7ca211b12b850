"""Textbook double-precision restatements used to pin the oracle.

Pure Python loops over lists (math.exp / math.sqrt), written without the
oracle's code or NumPy's matmul, so that a slip in the oracle (a dropped
term, a wrong sign or index, a transposed operand) shows up as a mismatch.
Only for tiny shapes: every loop is explicit.
"""
from __future__ import annotations

import math
import struct


def bf16(x: float) -> float:
    """Round a Python float to fp32, then to bf16 (nearest, ties to even)."""
    (u,) = struct.unpack("<I", struct.pack("<f", x))
    lsb = (u >> 16) & 1
    u = ((u + 0x7FFF + lsb) >> 16) << 16
    (y,) = struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))
    return y


def dot(a, b):
    s = 0.0
    for i in range(len(a)):
        s += a[i] * b[i]
    return s


def matvec(W, x):
    """y[o] = sum_i W[o][i] * x[i]  (W stored [out][in])."""
    return [dot(W[o], x) for o in range(len(W))]


def softmax(s):
    m = max(s)
    e = [math.exp(v - m) for v in s]
    z = sum(e)
    return [v / z for v in e]


def attention_one_query(q, keys, values):
    """softmax(q.k / sqrt(D)) weighted sum of values, one query."""
    D = len(q)
    sc = [dot(q, k) / math.sqrt(D) for k in keys]
    p = softmax(sc)
    out = [0.0] * D
    for j in range(len(keys)):
        for d in range(D):
            out[d] += p[j] * values[j][d]
    return out


def block_attention(q, k_blk, v_blk, k_ctx, v_ctx):
    """q [S][Hq][D]; k_blk/v_blk [S][Hkv][D]; k_ctx/v_ctx [Hkv][T][D] -> [S][Hq][D].

    Every query sees all T context keys and all S block keys (no mask);
    query head h uses kv head h // (Hq // Hkv).
    """
    S, Hq = len(q), len(q[0])
    Hkv = len(k_blk[0])
    G = Hq // Hkv
    out = []
    for i in range(S):
        row = []
        for h in range(Hq):
            c = h // G
            keys = [k_ctx[c][t] for t in range(len(k_ctx[c]))] + [k_blk[j][c] for j in range(S)]
            vals = [v_ctx[c][t] for t in range(len(v_ctx[c]))] + [v_blk[j][c] for j in range(S)]
            row.append(attention_one_query(q[i][h], keys, vals))
        out.append(row)
    return out


def rmsnorm(x, g, eps):
    ms = sum(v * v for v in x) / len(x)
    r = 1.0 / math.sqrt(ms + eps)
    return [x[i] * r * g[i] for i in range(len(x))]


def silu(x):
    return x / (1.0 + math.exp(-x))


def confidence_argmax(logits):
    """Largest softmax probability and the first index of the largest logit."""
    m = max(logits)
    arg = logits.index(m)
    z = sum(math.exp(v - m) for v in logits)
    return 1.0 / z, arg


def denoise_step(cfg, w, k_ctx, v_ctx, tokens, mask, round_act=False):
    """One denoising step before the commit rule: returns (logits [B*S][V], conf, arg).

    w: dict of nested lists (same names as the synthetic weight set).
    k_ctx/v_ctx: [L][B][Hkv][T][D] nested lists.
    round_act: store the GEMM inputs, q/k/v, attention output and SwiGLU
    product in bf16, like a bf16 model.
    """
    st = bf16 if round_act else (lambda v: v)
    B, S, H = cfg.batch, cfg.block, cfg.hidden
    Hq, Hkv, D, V = cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.vocab
    xs = []
    for b in range(B):
        for i in range(S):
            tid = V if (mask[b] >> i) & 1 else tokens[b][i]
            xs.append([w["embed"][tid][c] + w["pos"][i][c] for c in range(H)])
    for l in range(cfg.n_layers):
        ys = [[st(v) for v in rmsnorm(x, w[f"g_attn{l}"], cfg.rms_eps)] for x in xs]
        qs = [matvec(w[f"wq{l}"], y) for y in ys]
        ks = [matvec(w[f"wk{l}"], y) for y in ys]
        theta = getattr(cfg, "rope_theta", 0.0)
        if theta > 0:
            T = len(k_ctx[l][0][0]) if k_ctx[l] and k_ctx[l][0] else 0
            qs = [rope_row(qs[r], T + r % S, Hq, D, theta) for r in range(len(qs))]
            ks = [rope_row(ks[r], T + r % S, Hkv, D, theta) for r in range(len(ks))]
        qs = [[st(v) for v in q] for q in qs]
        ks = [[st(v) for v in k] for k in ks]
        vs = [[st(v) for v in matvec(w[f"wv{l}"], y)] for y in ys]
        new_xs = []
        for b in range(B):
            q = [[qs[b * S + i][h * D:(h + 1) * D] for h in range(Hq)] for i in range(S)]
            kb = [[ks[b * S + i][c * D:(c + 1) * D] for c in range(Hkv)] for i in range(S)]
            vb = [[vs[b * S + i][c * D:(c + 1) * D] for c in range(Hkv)] for i in range(S)]
            o = block_attention(q, kb, vb, k_ctx[l][b], v_ctx[l][b])
            for i in range(S):
                flat = [st(o[i][h][d]) for h in range(Hq) for d in range(D)]
                proj = matvec(w[f"wo{l}"], flat)
                new_xs.append([xs[b * S + i][c] + proj[c] for c in range(H)])
        xs = new_xs
        new_xs = []
        for x in xs:
            y = [st(v) for v in rmsnorm(x, w[f"g_mlp{l}"], cfg.rms_eps)]
            gt = matvec(w[f"wg{l}"], y)
            up = matvec(w[f"wu{l}"], y)
            hm = [st(silu(gt[f]) * up[f]) for f in range(len(gt))]
            dn = matvec(w[f"wd{l}"], hm)
            new_xs.append([x[c] + dn[c] for c in range(H)])
        xs = new_xs
    logits, conf, arg = [], [], []
    for x in xs:
        y = [st(v) for v in rmsnorm(x, w["g_final"], cfg.rms_eps)]
        lg = matvec(w["lm_head"], y)
        c, a = confidence_argmax(lg)
        logits.append(lg)
        conf.append(c)
        arg.append(a)
    return logits, conf, arg


def rope_row(x, pos, heads, D, theta):
    """Rotate the pairs (2j, 2j+1) of every head of one row by pos * theta^(-2j/D)."""
    out = list(x)
    for h in range(heads):
        for j in range(D // 2):
            a = pos * theta ** (-2.0 * j / D)
            c, s = math.cos(a), math.sin(a)
            e, o = x[h * D + 2 * j], x[h * D + 2 * j + 1]
            out[h * D + 2 * j] = e * c - o * s
            out[h * D + 2 * j + 1] = e * s + o * c
    return out


def commit_sets(conf_row, masked, gamma, mock_ar):
    """The set of positions committed for one sequence, stated as sets.

    All masked positions whose confidence reaches gamma; if that set is
    empty, the masked positions of highest confidence, of which the lowest;
    in mock-AR mode, the lowest masked position.
    """
    masked = set(masked)
    if not masked:
        return set()
    if mock_ar:
        return {min(masked)}
    hit = {i for i in masked if conf_row[i] >= gamma}
    if hit:
        return hit
    top = max(conf_row[i] for i in masked)
    return {min(i for i in masked if conf_row[i] == top)}


def top2_gap(row):
    """Largest value of a list minus the second largest (0 on an exact tie)."""
    a = sorted(row, reverse=True)
    return a[0] - a[1]


def near_tie_positions(rows, conf, masked, gamma, kind, k=0):
    """The near-tie positions of one sequence, stated as sets.

    rows[i]: logit row of position i; conf[i]: its confidence; masked: the
    masked positions; kind: "threshold", "mock_ar" or "cut" (top-k and
    fixed steps, k = positions to commit).  A masked position is a near-tie
    when its top-2 logit gap is below 1e-2; in threshold mode also when its
    confidence is within 1e-3 of gamma, or, when no masked confidence reaches
    gamma, when two masked confidences lie within 1e-3 of the largest one
    and it is one of them; in the cut modes when the k-th and (k+1)-th
    largest masked confidences are within 1e-3 and its confidence is within
    1e-3 of either.
    """
    masked = sorted(set(masked))
    out = {i for i in masked if top2_gap(rows[i]) < 1e-2}
    if not masked:
        return out
    ranked = sorted((conf[i] for i in masked), reverse=True)
    if kind == "threshold":
        out |= {i for i in masked if abs(conf[i] - gamma) < 1e-3}
        if all(conf[i] < gamma for i in masked):
            near_top = {i for i in masked if ranked[0] - conf[i] < 1e-3}
            if len(near_top) > 1:
                out |= near_top
    elif kind == "cut" and 0 < k < len(masked):
        a, b = ranked[k - 1], ranked[k]
        if a - b < 1e-3:
            out |= {i for i in masked if abs(conf[i] - a) < 1e-3 or abs(conf[i] - b) < 1e-3}
    return out


def tower_kv(tw, tokens, eps, n_layers, Hkv, D):
    """The context tower's K/V for one committed block, pure Python:
    returns kv[l][i] = the 2*Hkv*D bf16-rounded values (K rows, then V rows)
    of position i for denoiser layer l.  One causal self-attention layer
    (position i sees positions j <= i), residual, RMSNorm, then the per-layer
    projections.  tw: nested lists with the names of the synthetic tower."""
    S = len(tokens)
    H = len(tw["ctx_g"])
    es = [list(tw["ctx_embed"][t]) for t in tokens]
    ys = [rmsnorm(e, tw["ctx_g"], eps) for e in es]
    qkv = [matvec(tw["ctx_wqkv"], y) for y in ys]
    W = Hkv * D
    zs = []
    for i in range(S):
        a = []
        for h in range(Hkv):
            q = qkv[i][h * D:(h + 1) * D]
            keys = [qkv[j][W + h * D:W + (h + 1) * D] for j in range(i + 1)]
            vals = [qkv[j][2 * W + h * D:2 * W + (h + 1) * D] for j in range(i + 1)]
            a += attention_one_query(q, keys, vals)
        o = matvec(tw["ctx_wo"], a)
        hrow = [es[i][c] + o[c] for c in range(H)]
        zs.append(rmsnorm(hrow, tw["ctx_g2"], eps))
    return [[[bf16(v) for v in matvec(tw["ctx_wkv"][l], zs[i])] for i in range(S)] for l in range(n_layers)]
