"""Pins for the CPU oracle: brute force, closed forms and invariants (no GPU)."""
import math

import numpy as np
import pytest

import oracle
import synth
from tests import bruteforce as bf

F32 = np.float32

# A micro workload small enough for the pure-Python brute force.
MICRO = synth.Config("micro", batch=2, block=4, hidden=16, n_q_heads=4, n_kv_heads=2,
                     head_dim=4, n_layers=2, mlp=24, vocab=32, ctx_len=5, max_ctx=5)


def _micro_model(cfg=MICRO, seed=3, lm_std=None):
    wb = synth.make_weights(cfg, seed)
    kb, vb = synth.make_context_kv(cfg, seed)
    return oracle.OracleModel.from_bits(cfg, wb, kb, vb, synth.bf16_bits_to_f32)


# ---------------------------------------------------------------- attention

@pytest.mark.parametrize("T,Hq,Hkv", [(0, 4, 4), (1, 4, 2), (17, 4, 1), (40, 2, 2)])
def test_attention_vs_bruteforce(T, Hq, Hkv):
    rng = np.random.default_rng(T * 7 + Hkv)
    S, D = 16, 8
    q = rng.standard_normal((S, Hq, D)).astype(F32) * 2
    kb = rng.standard_normal((S, Hkv, D)).astype(F32)
    vb = rng.standard_normal((S, Hkv, D)).astype(F32)
    kc = rng.standard_normal((Hkv, T, D)).astype(F32)
    vc = rng.standard_normal((Hkv, T, D)).astype(F32)
    got = oracle.block_attention(q, kb, vb, kc, vc)
    ref = np.array(bf.block_attention(q.tolist(), kb.tolist(), vb.tolist(), kc.tolist(), vc.tolist()))
    np.testing.assert_allclose(got, ref, rtol=2e-5, atol=2e-6)


def test_attention_constant_values():
    """Constant value rows give that constant whatever the scores."""
    rng = np.random.default_rng(1)
    S, Hq, Hkv, D, T = 16, 4, 2, 8, 33
    q = rng.standard_normal((S, Hq, D)).astype(F32) * 3
    kb = rng.standard_normal((S, Hkv, D)).astype(F32)
    kc = rng.standard_normal((Hkv, T, D)).astype(F32)
    c = rng.standard_normal((Hkv, D)).astype(F32)
    vb = np.broadcast_to(c[None], (S, Hkv, D)).copy()
    vc = np.broadcast_to(c[:, None], (Hkv, T, D)).copy()
    out = oracle.block_attention(q, kb, vb, kc, vc)
    for h in range(Hq):
        np.testing.assert_allclose(out[:, h], np.broadcast_to(c[h // 2], (S, D)), rtol=1e-5, atol=1e-6)


def test_attention_zero_query_is_uniform_mean():
    """q = 0 makes every score equal: the output is the mean of all T+S values."""
    rng = np.random.default_rng(2)
    S, Hq, Hkv, D, T = 16, 2, 1, 8, 9
    q = np.zeros((S, Hq, D), F32)
    kb = rng.standard_normal((S, Hkv, D)).astype(F32)
    vb = rng.standard_normal((S, Hkv, D)).astype(F32)
    kc = rng.standard_normal((Hkv, T, D)).astype(F32)
    vc = rng.standard_normal((Hkv, T, D)).astype(F32)
    out = oracle.block_attention(q, kb, vb, kc, vc)
    mean = np.concatenate([vc[0], vb[:, 0]]).mean(axis=0)
    np.testing.assert_allclose(out[:, 0], np.broadcast_to(mean, (S, D)), rtol=1e-5, atol=1e-6)


def test_attention_gqa_equals_repeated_mha():
    """GQA with G query heads per kv head equals MHA with each kv head repeated G times."""
    rng = np.random.default_rng(3)
    S, Hq, Hkv, D, T = 16, 8, 2, 8, 12
    q = rng.standard_normal((S, Hq, D)).astype(F32)
    kb = rng.standard_normal((S, Hkv, D)).astype(F32)
    vb = rng.standard_normal((S, Hkv, D)).astype(F32)
    kc = rng.standard_normal((Hkv, T, D)).astype(F32)
    vc = rng.standard_normal((Hkv, T, D)).astype(F32)
    gqa = oracle.block_attention(q, kb, vb, kc, vc)
    rep = lambda a, ax: np.repeat(a, Hq // Hkv, axis=ax)
    mha = oracle.block_attention(q, rep(kb, 1), rep(vb, 1), rep(kc, 0), rep(vc, 0))
    np.testing.assert_allclose(gqa, mha, rtol=1e-6, atol=1e-7)


def test_attention_is_bidirectional_and_sees_context():
    """Changing the LAST block key changes the FIRST query's output (no causal
    mask), and changing one context value changes every query's output."""
    rng = np.random.default_rng(4)
    S, Hq, Hkv, D, T = 16, 2, 2, 8, 6
    q = rng.standard_normal((S, Hq, D)).astype(F32)
    kb = rng.standard_normal((S, Hkv, D)).astype(F32)
    vb = rng.standard_normal((S, Hkv, D)).astype(F32)
    kc = rng.standard_normal((Hkv, T, D)).astype(F32)
    vc = rng.standard_normal((Hkv, T, D)).astype(F32)
    base = oracle.block_attention(q, kb, vb, kc, vc)
    vb2 = vb.copy()
    vb2[-1] += 5
    assert np.abs(oracle.block_attention(q, kb, vb2, kc, vc)[0] - base[0]).max() > 1e-4
    vc2 = vc.copy()
    vc2[:, 0] += 5
    assert np.all(np.abs(oracle.block_attention(q, kb, vb, kc, vc2) - base).max(axis=2) > 1e-5)


# ---------------------------------------------------------- confidence select

def test_select_equal_logits():
    V = 4096
    conf, arg = oracle.select_from_logits(np.full((3, V), 1.25, F32))
    np.testing.assert_allclose(conf, 1.0 / V, rtol=1e-5)
    assert (arg == 0).all()


@pytest.mark.parametrize("delta", [0.5, 3.0, 9.0])
def test_select_single_lead_closed_form(delta):
    V, lead = 1000, 417
    lg = np.zeros((1, V), F32)
    lg[0, lead] = delta
    conf, arg = oracle.select_from_logits(lg)
    assert arg[0] == lead
    np.testing.assert_allclose(conf[0], 1.0 / (1.0 + (V - 1) * math.exp(-delta)), rtol=1e-5)


def test_select_vs_bruteforce_and_first_max():
    rng = np.random.default_rng(5)
    lg = (rng.standard_normal((6, 300)) * 8).astype(F32)
    lg[2, 10] = lg[2, 250] = lg[2].max() + 1.0            # tie: lowest id wins
    conf, arg = oracle.select_from_logits(lg)
    for r in range(lg.shape[0]):
        c, a = bf.confidence_argmax(lg[r].astype(np.float64).tolist())
        assert arg[r] == a
        assert abs(conf[r] - c) <= 1e-5 * c
    assert arg[2] == 10


# ---------------------------------------------------------------- norm / MLP

def test_rmsnorm_closed_forms():
    H = 64
    g = np.linspace(0.5, 1.5, H).astype(F32)
    x = np.full((1, H), 3.0, F32)
    np.testing.assert_allclose(oracle.rmsnorm(x, g, 1e-5)[0], 3.0 / math.sqrt(9.0 + 1e-5) * g, rtol=1e-6)
    rng = np.random.default_rng(6)
    x = rng.standard_normal((4, H)).astype(F32)
    y1 = oracle.rmsnorm(x, g, 0.0)
    y2 = oracle.rmsnorm(x * 37.0, g, 0.0)
    np.testing.assert_allclose(y1, y2, rtol=1e-5, atol=1e-6)
    for r in range(4):
        np.testing.assert_allclose(y1[r], bf.rmsnorm(x[r].tolist(), g.tolist(), 0.0), rtol=1e-5, atol=1e-6)


def test_silu_values():
    x = np.array([0.0, 1.0, -1.0, 20.0, -20.0], F32)
    ref = np.array([0.0, 1 / (1 + math.exp(-1)), -1 / (1 + math.exp(1)), 20.0, -20 / (1 + math.exp(20))])
    np.testing.assert_allclose(oracle.silu(x), ref, rtol=1e-6, atol=1e-12)


def test_round_bf16_matches_bruteforce():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(2000) * np.exp(rng.uniform(-20, 20, 2000))).astype(F32)
    x[:4] = [1.00390625, 1.01171875, -1.00390625, 0.0]      # exact ties -> even
    got = oracle.round_bf16(x)
    ref = np.array([bf.bf16(float(v)) for v in x], F32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert got[0] == 1.0 and got[1] == 1.015625


# ---------------------------------------------------------------- full step

def _nested(a):
    return a.tolist()


@pytest.mark.parametrize("round_act", [False, True])
def test_full_step_vs_bruteforce(round_act):
    cfg = MICRO
    m = _micro_model(cfg)
    tok, mask = synth.make_tokens(cfg, seed=1, masked_frac=0.6)
    r = oracle.denoise_step(m, tok, mask, 0.8, act_bf16=round_act, keep_intermediates=True)
    w = {k: _nested(v) for k, v in m.w.items()}
    logits, conf, arg = bf.denoise_step(cfg, w, _nested(m.k_ctx), _nested(m.v_ctx),
                                        tok.tolist(), [int(v) for v in mask], round_act)
    tol = 1e-2 if round_act else 2e-4
    np.testing.assert_allclose(r.logits, np.array(logits), rtol=tol, atol=tol * 0.1)
    np.testing.assert_allclose(r.conf.reshape(-1), np.array(conf), rtol=tol, atol=1e-6)
    assert (r.arg.reshape(-1) == np.array(arg)).all()


def test_full_step_vs_bruteforce_random_gains():
    """Non-unit RMSNorm gains, so a gain applied at the wrong norm shows."""
    cfg = MICRO
    m = _micro_model(cfg)
    rng = np.random.default_rng(11)
    for name in list(m.w):
        if name.startswith("g_"):
            m.w[name] = oracle.round_bf16((1.0 + 0.4 * rng.standard_normal(m.w[name].shape)).astype(F32))
    tok, mask = synth.make_tokens(cfg, seed=4, masked_frac=0.5)
    r = oracle.denoise_step(m, tok, mask, 0.8, keep_intermediates=True)
    w = {k: _nested(v) for k, v in m.w.items()}
    logits, conf, arg = bf.denoise_step(cfg, w, _nested(m.k_ctx), _nested(m.v_ctx),
                                        tok.tolist(), [int(v) for v in mask], False)
    np.testing.assert_allclose(r.logits, np.array(logits), rtol=2e-4, atol=2e-5)
    assert (r.arg.reshape(-1) == np.array(arg)).all()


def test_bf16_storage_alone_moves_logits():
    """Storing activations in bf16 (a bf16 model's dataflow) moves the tiny
    workload's logits by far more than the 2e-2 parity bar: the reason the
    reference keeps activations in fp32."""
    cfg = synth.TINY
    m = oracle.OracleModel.from_bits(cfg, synth.make_weights(cfg, 0), *synth.make_context_kv(cfg, 0),
                                     synth.bf16_bits_to_f32)
    tok, mask = synth.make_tokens(cfg, seed=0)
    a = oracle.denoise_step(m, tok, mask, 0.8, act_bf16=False, keep_intermediates=True)
    b = oracle.denoise_step(m, tok, mask, 0.8, act_bf16=True, keep_intermediates=True)
    assert np.abs(a.logits - b.logits).max() > 5e-2


def test_full_step_linear_in_lm_head_scale():
    """Scaling the LM head by c scales the logits by c exactly up to rounding."""
    m = _micro_model()
    tok, mask = synth.make_tokens(MICRO, seed=2)
    r1 = oracle.denoise_step(m, tok, mask, 0.8, act_bf16=False, keep_intermediates=True)
    m.w["lm_head"] = m.w["lm_head"] * F32(4.0)
    r2 = oracle.denoise_step(m, tok, mask, 0.8, act_bf16=False, keep_intermediates=True)
    np.testing.assert_allclose(r2.logits, 4 * r1.logits, rtol=1e-6, atol=1e-6)


# ------------------------------------------------------------- commit rule

def test_commit_exhaustive_masks():
    """Every mask of a 16-position block, two crafted confidence rows, both modes,
    against the set-based statement of the rule."""
    S = 16
    rows = [np.array([0.1, 0.85, 0.3, 0.8, 0.79, 0.95, 0.2, 0.8, 0.5, 0.99, 0.01, 0.6,
                      0.7, 0.81, 0.4, 0.3], F32),
            np.array([0.5, 0.7, 0.7, 0.1, 0.2, 0.7, 0.3, 0.6, 0.1, 0.2, 0.3, 0.4,
                      0.5, 0.6, 0.7, 0.05], F32)]
    masks = np.arange(1, 1 << S, dtype=np.uint32)
    for conf in rows:
        arg = (np.arange(S, dtype=np.int32) * 97 + 5)[None]
        for mode in (oracle.MODE_THRESHOLD, oracle.MODE_MOCK_AR):
            B = len(masks)
            toks = np.full((B, S), 4096, np.int32)
            new_tok, new_mask, n, _ = oracle.commit(np.broadcast_to(conf, (B, S)),
                                                    np.broadcast_to(arg, (B, S)), toks, masks,
                                                    0.8, mode, S)
            for b in range(0, B, 7):             # every 7th mask keeps this to seconds
                mk = int(masks[b])
                masked = [i for i in range(S) if (mk >> i) & 1]
                want = bf.commit_sets(conf.tolist(), masked, F32(0.8), mode == oracle.MODE_MOCK_AR)
                got = {i for i in range(S) if (mk >> i) & 1 and not (int(new_mask[b]) >> i) & 1}
                assert got == want, (mk, mode)
                assert n[b] == len(want)
                for i in range(S):
                    assert new_tok[b, i] == (arg[0, i] if i in want else 4096)


def test_commit_gamma_zero_and_above_one():
    rng = np.random.default_rng(8)
    conf = rng.uniform(0, 1, (5, 16)).astype(F32)
    arg = rng.integers(0, 100, (5, 16)).astype(np.int32)
    tok = np.full((5, 16), 100, np.int32)
    mask = np.array([0xFFFF, 0x0F0F, 0x8001, 0x1, 0x7FFE], np.uint32)
    _, m0, n0, _ = oracle.commit(conf, arg, tok, mask, 0.0, oracle.MODE_THRESHOLD, 16)
    assert (m0 == 0).all() and list(n0) == [bin(int(v)).count("1") for v in mask]
    _, m2, n2, fb = oracle.commit(conf, arg, tok, mask, 1.5, oracle.MODE_THRESHOLD, 16)
    assert (n2 == 1).all() and fb.all()
    for b in range(5):
        gone = int(mask[b]) & ~int(m2[b])
        i = gone.bit_length() - 1
        masked = [j for j in range(16) if (int(mask[b]) >> j) & 1]
        assert conf[b, i] == max(conf[b, j] for j in masked)


def test_commit_monotone_in_gamma():
    rng = np.random.default_rng(9)
    conf = rng.uniform(0, 1, (64, 16)).astype(F32)
    arg = np.zeros((64, 16), np.int32)
    tok = np.zeros((64, 16), np.int32)
    mask = rng.integers(1, 1 << 16, 64).astype(np.uint32)
    prev = None
    for g in (0.1, 0.3, 0.5, 0.8, 0.95):
        _, m, _, fb = oracle.commit(conf, arg, tok, mask, g, oracle.MODE_THRESHOLD, 16)
        done = mask & ~m
        if prev is not None:
            # a larger gamma commits a subset, unless the fallback picked its one position
            ok = ((done & ~prev) == 0) | fb
            assert ok.all()
        prev = done


# ------------------------------------------------------------- near-ties

NEAR_TIE_MODES = ([(0.8, oracle.MODE_THRESHOLD), (0.5, oracle.MODE_THRESHOLD), (0.8, oracle.MODE_MOCK_AR)]
                  + [(0.8, oracle.with_param(oracle.MODE_TOPK, k)) for k in (1, 2, 3, 5)]
                  + [(0.8, oracle.with_param(oracle.MODE_STEPS, n)) for n in (2, 4, 7)])


def _near_tie_dense(seed, B=48, S=16, V=6, gamma=0.8):
    """Logits, confidences and masks crowded with near-ties: a third of the
    logit rows have a top-2 gap under 2e-2, and confidences cluster within
    2e-3 of a few anchors (gamma among them)."""
    rng = np.random.default_rng(seed)
    logits = rng.normal(0, 1, (B * S, V)).astype(F32)
    close_rows = rng.random(B * S) < 0.35
    top = logits.argmax(axis=1)
    second = (top + 1 + rng.integers(0, V - 1, B * S)) % V
    gap = rng.uniform(0, 0.02, B * S).astype(F32)
    logits[np.arange(B * S), second] = np.where(close_rows, logits[np.arange(B * S), top] - gap,
                                                logits[np.arange(B * S), second])
    anchors = np.array([gamma, 0.5, 0.62, 0.3, 0.95, 0.7], F32)
    conf = (anchors[rng.integers(0, anchors.size, (B, S))] + rng.uniform(-2e-3, 2e-3, (B, S))).astype(F32)
    mask = rng.integers(1, 1 << S, B).astype(np.uint32)
    return logits, conf, mask


@pytest.mark.parametrize("gamma,mode", NEAR_TIE_MODES)
def test_near_tie_positions_vs_bruteforce(gamma, mode):
    """The oracle's near-tie flags equal the set statement in tests/bruteforce.py."""
    S = 16
    logits, conf, mask = _near_tie_dense(11, gamma=gamma)
    flags = oracle.near_tie_positions(logits, conf, mask, gamma, mode, S)
    base, param = mode & 0xFF, mode >> 8
    for b in range(mask.size):
        masked = [i for i in range(S) if (int(mask[b]) >> i) & 1]
        rows = [logits[b * S + i].astype(np.float64).tolist() for i in range(S)]
        c = [float(v) for v in conf[b]]
        if base == oracle.MODE_THRESHOLD:
            want = bf.near_tie_positions(rows, c, masked, float(F32(gamma)), "threshold")
        elif base == oracle.MODE_MOCK_AR:
            want = bf.near_tie_positions(rows, c, masked, gamma, "mock_ar")
        else:
            k = param if base == oracle.MODE_TOPK else oracle.steps_schedule_k(S, param, len(masked))
            want = bf.near_tie_positions(rows, c, masked, gamma, "cut", k)
        assert set(np.nonzero(flags[b])[0].tolist()) == want, (b, hex(int(mask[b])))


@pytest.mark.parametrize("gamma,mode", NEAR_TIE_MODES)
def test_near_tie_flags_are_sound(gamma, mode):
    """What the flags promise: perturbing every logit by less than half the
    logit-gap bound and every confidence by less than half the confidence
    bounds changes the committed ids and mask only at flagged positions."""
    S = 16
    logits, conf, mask = _near_tie_dense(12, gamma=gamma)
    B = mask.size
    flags = oracle.near_tie_positions(logits, conf, mask, gamma, mode, S)
    tok0 = np.full((B, S), 1 << 20, np.int32)
    arg = logits.argmax(axis=1).astype(np.int32).reshape(B, S)
    t_ref, m_ref, _, _ = oracle.commit(conf, arg, tok0, mask, gamma, mode, S)
    bits = (m_ref[:, None] >> np.arange(S)) & 1
    rng = np.random.default_rng(13)
    changed = 0
    for _ in range(150):
        lp = logits + rng.uniform(-4.9e-3, 4.9e-3, logits.shape).astype(F32)
        cp = (conf + rng.uniform(-4.9e-4, 4.9e-4, conf.shape)).astype(F32)
        ap = lp.argmax(axis=1).astype(np.int32).reshape(B, S)
        t, m, _, _ = oracle.commit(cp, ap, tok0, mask, gamma, mode, S)
        diff = (t != t_ref) | ((((m[:, None] >> np.arange(S)) & 1) != bits))
        assert not (diff & ~flags).any(), np.argwhere(diff & ~flags)[:5]
        changed += int(diff.any())
    if mode & 0xFF != oracle.MODE_MOCK_AR:
        assert changed > 0   # the data does sit on near-ties


# ------------------------------------------------------- decode invariants

@pytest.fixture(scope="module")
def tiny_model():
    cfg = synth.TINY.replace(batch=2, ctx_len=64, max_ctx=64)
    wb = synth.make_weights(cfg, 0)
    kb, vb = synth.make_context_kv(cfg, 0)
    return oracle.OracleModel.from_bits(cfg, wb, kb, vb, synth.bf16_bits_to_f32)


def test_decode_gamma_zero_fills_in_one_step(tiny_model):
    tok, steps, hist = oracle.decode_block(tiny_model, 0.0)
    assert steps == 1 and (hist[0] == 16).all()


def test_decode_gamma_above_one_takes_block_steps(tiny_model):
    tok, steps, hist = oracle.decode_block(tiny_model, 1.01)
    assert steps == 16 and all((h == 1).all() for h in hist)


def test_decode_mock_ar_is_left_to_right(tiny_model):
    cfg = tiny_model.cfg
    tokens = np.full((cfg.batch, 16), cfg.vocab, np.int32)
    mask = np.full(cfg.batch, 0xFFFF, np.uint32)
    for step in range(16):
        r = oracle.denoise_step(tiny_model, tokens, mask, 0.8, oracle.MODE_MOCK_AR)
        assert (r.mask == (0xFFFF & ~((1 << (step + 1)) - 1))).all()
        tokens, mask = r.tokens, r.mask


def test_decode_committed_never_change_and_progress(tiny_model):
    cfg = tiny_model.cfg
    tokens = np.full((cfg.batch, 16), cfg.vocab, np.int32)
    mask = np.full(cfg.batch, 0xFFFF, np.uint32)
    while mask.max():
        r = oracle.denoise_step(tiny_model, tokens, mask, 0.8)
        for b in range(cfg.batch):
            if mask[b]:
                assert r.n_committed[b] >= 1
            for i in range(16):
                if not (int(mask[b]) >> i) & 1:
                    assert r.tokens[b, i] == tokens[b, i]
            assert int(r.mask[b]) & ~int(mask[b]) == 0
        tokens, mask = r.tokens, r.mask
    assert (tokens < cfg.vocab).all()


def test_batch_independence(tiny_model):
    """Sequence b decoded in a batch equals sequence b decoded alone."""
    cfg = tiny_model.cfg
    tok_all, _, _ = oracle.decode_block(tiny_model, 0.8)
    for b in range(cfg.batch):
        one = oracle.OracleModel(cfg.replace(batch=1), tiny_model.w,
                                 tiny_model.k_ctx[:, b:b + 1], tiny_model.v_ctx[:, b:b + 1],
                                 tiny_model.ctx_len)
        tok_one, _, _ = oracle.decode_block(one, 0.8)
        assert (tok_one[0] == tok_all[b]).all()


# ------------------------------------------------- top-k and fixed steps

def test_commit_topk_exhaustive_masks():
    """Top-k over every mask of a 16-position block: the committed set is the
    k masked positions that precede every other masked position in the order
    (higher confidence first, lower position on equal confidence)."""
    S = 16
    conf = np.array([[0.5, 0.9, 0.1, 0.9, 0.3, 0.7, 0.7, 0.2, 0.05, 0.6, 0.9, 0.4, 0.35, 0.8, 0.15, 0.7]], F32)
    arg = np.arange(S, dtype=np.int32).reshape(1, S) + 1000
    for k in (1, 3, 16):
        mode = oracle.with_param(oracle.MODE_TOPK, k)
        for mk in range(1 << S):
            tok0 = np.zeros((1, S), np.int32)
            tok, m, n, _ = oracle.commit(conf, arg, tok0, np.array([mk], np.uint32), 0.8, mode, S)
            masked = [i for i in range(S) if (mk >> i) & 1]
            chosen = [i for i in masked if not (int(m[0]) >> i) & 1]
            assert len(chosen) == min(k, len(masked)) and int(n[0]) == len(chosen)
            rest = [j for j in masked if j not in chosen]
            for i in chosen:
                assert tok[0, i] == 1000 + i
                for j in rest:
                    assert conf[0, i] > conf[0, j] or (conf[0, i] == conf[0, j] and i < j)


@pytest.mark.parametrize("S", [1, 5, 16, 32])
def test_steps_schedule_fills_block_in_n_steps(S):
    for N in range(1, S + 4):
        left, steps = S, 0
        while left:
            k = oracle.steps_schedule_k(S, N, left)
            assert 1 <= k <= left
            left -= k
            steps += 1
        assert steps == min(N, S)


def test_decode_topk_and_fixed_steps(tiny_model):
    _, steps, hist = oracle.decode_block(tiny_model, 0.8, oracle.with_param(oracle.MODE_TOPK, 3))
    assert steps == 6 and all((h == 3).all() for h in hist[:5]) and (hist[5] == 1).all()
    for N in (1, 5, 16):
        _, steps, _ = oracle.decode_block(tiny_model, 0.8, oracle.with_param(oracle.MODE_STEPS, N))
        assert steps == N


def test_decode_top1_equals_gamma_above_one(tiny_model):
    """Top-1 commits the single most confident masked position every step,
    which is what the threshold rule does when no confidence can reach gamma."""
    a, sa, _ = oracle.decode_block(tiny_model, 0.8, oracle.with_param(oracle.MODE_TOPK, 1))
    b, sb, _ = oracle.decode_block(tiny_model, 1.01)
    assert sa == sb == 16 and (a == b).all()


# ------------------------------------------------------------------- RoPE

def test_rope_closed_forms():
    x = np.zeros((3, 1, 2), F32)
    x[:, 0, 0] = 1.0
    got = oracle.rope(x, np.array([0, 1, 2]), 10000.0)       # D = 2: frequency theta^0 = 1
    np.testing.assert_allclose(got[:, 0, 0], np.cos([0.0, 1.0, 2.0]), atol=1e-7)
    np.testing.assert_allclose(got[:, 0, 1], np.sin([0.0, 1.0, 2.0]), atol=1e-7)
    rng = np.random.default_rng(12)
    y = rng.standard_normal((5, 3, 16)).astype(F32)
    r = oracle.rope(y, np.arange(5) * 37 + 3, 500.0)
    np.testing.assert_allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(y, axis=-1), rtol=1e-5)
    np.testing.assert_array_equal(oracle.rope(y, np.zeros(5, int), 500.0), y)


def test_rope_scores_depend_on_relative_position():
    rng = np.random.default_rng(13)
    q = rng.standard_normal((4, 2, 8)).astype(F32)
    k = rng.standard_normal((4, 2, 8)).astype(F32)
    pos = np.array([0, 3, 7, 20])
    for shift in (1, 50, 1000):
        a = np.einsum("ihd,jhd->hij", oracle.rope(q, pos, 100.0), oracle.rope(k, pos, 100.0))
        b = np.einsum("ihd,jhd->hij", oracle.rope(q, pos + shift, 100.0), oracle.rope(k, pos + shift, 100.0))
        np.testing.assert_allclose(a, b, rtol=1e-4, atol=1e-4)


def test_full_step_with_rope_vs_bruteforce():
    cfg = MICRO.replace(rope_theta=100.0)
    m = _micro_model(cfg)
    tok, mask = synth.make_tokens(cfg, seed=5, masked_frac=0.5)
    r = oracle.denoise_step(m, tok, mask, 0.8, keep_intermediates=True)
    w = {k: _nested(v) for k, v in m.w.items()}
    logits, conf, arg = bf.denoise_step(cfg, w, _nested(m.k_ctx), _nested(m.v_ctx),
                                        tok.tolist(), [int(v) for v in mask], False)
    np.testing.assert_allclose(r.logits, np.array(logits), rtol=2e-4, atol=2e-5)
    assert (r.arg.reshape(-1) == np.array(arg)).all()
    plain = oracle.denoise_step(_micro_model(MICRO), tok, mask, 0.8, keep_intermediates=True)
    assert np.abs(plain.logits - r.logits).max() > 1e-3   # the rotation reaches the logits


# ------------------------------------------------- context tower (append)

def _tower(cfg, seed=0):
    return {k: synth.bf16_bits_to_f32(v) for k, v in synth.make_tower_weights(cfg, seed).items()}


def test_append_block_vs_bruteforce():
    cfg = MICRO
    m = _micro_model(cfg)
    tw = _tower(cfg)
    rng = np.random.default_rng(14)
    for g in ("ctx_g", "ctx_g2"):        # non-unit gains, so each norm's gain is checked
        tw[g] = oracle.round_bf16(rng.normal(1.0, 0.3, cfg.hidden).astype(F32))
    tok = rng.integers(0, cfg.vocab, (cfg.batch, cfg.block)).astype(np.int32)
    tok[0, 1] = tok[0, 3]                                         # a repeated token
    m2 = oracle.append_block(m, tw, tok)
    T, S, Hkv, D = m.ctx_len, cfg.block, cfg.n_kv_heads, cfg.head_dim
    assert m2.ctx_len == T + S
    np.testing.assert_array_equal(m2.k_ctx[:, :, :, :T], m.k_ctx[:, :, :, :T])
    np.testing.assert_array_equal(m2.v_ctx[:, :, :, :T], m.v_ctx[:, :, :, :T])
    twl = {k: v.tolist() for k, v in tw.items()}
    for b in range(cfg.batch):
        kv = bf.tower_kv(twl, tok[b].tolist(), cfg.rms_eps, cfg.n_layers, Hkv, D)
        for l in range(cfg.n_layers):
            for i in range(S):
                for h in range(Hkv):
                    want_k = np.array(kv[l][i][h * D:(h + 1) * D], F32)
                    want_v = np.array(kv[l][i][Hkv * D + h * D:Hkv * D + (h + 1) * D], F32)
                    # one bf16 rounding apart at most (fp32 vs double before the rounding)
                    assert (np.abs(m2.k_ctx[l, b, h, T + i] - want_k) <= np.abs(want_k) * 2.0 ** -7 + 1e-30).all()
                    assert (np.abs(m2.v_ctx[l, b, h, T + i] - want_v) <= np.abs(want_v) * 2.0 ** -7 + 1e-30).all()
    # the repeated token sits at positions 1 and 3 but sees different prefixes
    assert not np.array_equal(m2.k_ctx[:, 0, :, T + 1], m2.k_ctx[:, 0, :, T + 3])


def test_append_block_is_causal():
    """Changing the committed token at position j changes the appended K/V of
    positions j and after, and of no position before j."""
    cfg = MICRO.replace(block=6, batch=1)
    m = _micro_model(cfg)
    tw = _tower(cfg)
    rng = np.random.default_rng(15)
    tok = rng.integers(0, cfg.vocab, (1, cfg.block)).astype(np.int32)
    base = oracle.append_block(m, tw, tok)
    T = m.ctx_len
    for j in range(cfg.block):
        t2 = tok.copy()
        t2[0, j] = (t2[0, j] + 1 + j) % cfg.vocab
        m2 = oracle.append_block(m, tw, t2)
        for i in range(cfg.block):
            same = (np.array_equal(m2.k_ctx[:, 0, :, T + i], base.k_ctx[:, 0, :, T + i]) and
                    np.array_equal(m2.v_ctx[:, 0, :, T + i], base.v_ctx[:, 0, :, T + i]))
            assert same == (i < j), (i, j)


def test_tower_attention_closed_forms():
    """Position 0 sees only itself (output = v_0); equal keys give the running
    mean of the values."""
    rng = np.random.default_rng(16)
    q = rng.standard_normal((5, 2, 4)).astype(F32)
    k = rng.standard_normal((5, 2, 4)).astype(F32)
    v = rng.standard_normal((5, 2, 4)).astype(F32)
    out = oracle.tower_causal_attention(q, k, v)
    np.testing.assert_allclose(out[0], v[0], rtol=1e-6)
    ke = np.broadcast_to(k[:1], k.shape).copy()
    out = oracle.tower_causal_attention(q, ke, v)
    for i in range(5):
        np.testing.assert_allclose(out[i], v[:i + 1].mean(axis=0), rtol=1e-5, atol=1e-6)


def test_decode_after_append_sees_the_new_context(tiny_model):
    cfg = tiny_model.cfg
    tw = _tower(cfg)
    tok, _, _ = oracle.decode_block(tiny_model, 0.8)
    m2 = oracle.append_block(tiny_model, tw, tok)
    start = np.full((cfg.batch, cfg.block), cfg.vocab, np.int32), np.full(cfg.batch, 0xFFFF, np.uint32)
    a = oracle.denoise_step(tiny_model, *start, 0.8, keep_intermediates=True)
    b = oracle.denoise_step(m2, *start, 0.8, keep_intermediates=True)
    assert np.abs(a.logits - b.logits).max() > 1e-4
