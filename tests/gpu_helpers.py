"""Shared set-up for the GPU parity tests: inputs from `synth`, the CUDA path
through the C-ABI, the expected values from `oracle`."""
from __future__ import annotations

import os

import numpy as np
import pytest

import oracle
import synth
from tests import near_tie_log

torch = pytest.importorskip("torch")

# Tolerances of the parity tests (abs and rel, |gpu - oracle| <= tol + tol*|oracle|).
TOL_ATTN = 1e-2
TOL_LOGIT = 2e-2
TOL_CONF = 2e-2


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_wise_masked_dd_b300 import build as libbuild
    libbuild.build()


def to_dev(bits: np.ndarray, device="cuda"):
    from block_wise_masked_dd_b300.decoder import bits_to_tensor
    return bits_to_tensor(bits, device)


def bf16_to_f32(t) -> np.ndarray:
    return t.float().cpu().numpy()


def close(got, want, tol, what="", rel_rms=None):
    """Elementwise |got - want| <= tol + tol*|want|; optionally also
    rms(got - want) <= rel_rms * rms(want) (catches small systematic drift
    that an absolute bound on small values would hide)."""
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    err = np.abs(got - want)
    bound = tol + tol * np.abs(want)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tol {tol}; worst at {i}: "
                             f"got {got[i]} want {want[i]}")
    if rel_rms is not None and err.size:
        r = np.sqrt(np.mean(err ** 2)) / max(np.sqrt(np.mean(want ** 2)), 1e-30)
        assert r <= rel_rms, f"{what}: relative rms error {r:.2e} > {rel_rms:.1e}"
    return float(err.max()) if err.size else 0.0


class Problem:
    """A synthetic decoding problem on both sides."""

    def __init__(self, cfg: synth.Config, seed: int = 0, device="cuda", key_growth: float = 0.0):
        """key_growth > 0 scales the context keys of 128-position tile t by
        1 + key_growth * t (then rounds them to bf16 again, for both sides):
        later tiles' scores then exceed the earlier maxima by far, which moves
        the attention kernels' reference maxima after the first tile."""
        from block_wise_masked_dd_b300.decoder import Decoder, pack_weights
        self.cfg = cfg
        self.w_bits = synth.make_weights(cfg, seed)
        self.k_bits, self.v_bits = synth.make_context_kv(cfg, seed)
        if key_growth:
            k = synth.bf16_bits_to_f32(self.k_bits)  # [L][B][Hkv][T][D]
            scale = 1.0 + key_growth * (np.arange(k.shape[3]) // 128)
            self.k_bits = synth.to_bf16_bits((k * scale[:, None]).astype(np.float32))
        self.model = oracle.OracleModel.from_bits(cfg, self.w_bits, self.k_bits, self.v_bits,
                                                  synth.bf16_bits_to_f32)
        self.weights = pack_weights(cfg, self.w_bits, device)
        self.dec = Decoder(cfg, self.weights, device)
        self.k_dev = to_dev(self.k_bits, device)
        self.v_dev = to_dev(self.v_bits, device)
        self.dec.set_context_kv(self.k_dev, self.v_dev, 0)
        torch.cuda.synchronize()

    def start_state(self):
        cfg = self.cfg
        tok = np.full((cfg.batch, cfg.block), cfg.vocab, np.int32)
        mask = np.full(cfg.batch, (1 << cfg.block) - 1, np.uint32)
        return tok, mask

    def gpu_state(self, tok, mask):
        t = torch.from_numpy(tok.copy()).cuda()
        m = torch.from_numpy(mask.view(np.int32).copy()).cuda()
        return t, m


def _masked_bits(mask, S):
    return ((np.asarray(mask, np.uint32)[:, None] >> np.arange(S)) & 1).astype(bool)


def check_commit(tok, mask, gamma, mode, S, r_tokens, r_mask, r_tie, g_tok, g_mask, g_n=None, r_n=None,
                 g_conf=None, g_arg=None, what="step"):
    """Token parity of one step taken by both sides from the same state
    (tok [B,S], mask [B]):

    * with the CUDA path's own confidences and ids (g_conf, g_arg, when
      given), its new ids, mask and counts are exactly the commit rule
      (`oracle.commit`) applied to them, in every sequence;
    * every position where the CUDA path and the oracle differ (committed
      id or mask bit) is a masked position the oracle flags as a near-tie;
      the counts agree in every sequence with no flagged position.

    Records and returns (flagged masked positions, masked positions)."""
    g_tok = np.asarray(g_tok)
    g_mask = np.asarray(g_mask, np.uint32)
    if g_conf is not None:
        e_tok, e_mask, e_n, _ = oracle.commit(np.asarray(g_conf, np.float32).reshape(-1, S),
                                              np.asarray(g_arg, np.int32).reshape(-1, S), tok, mask, gamma, mode, S)
        assert (g_mask == e_mask).all(), f"{what}: mask is not the commit rule on the CUDA path's own confidences"
        assert (g_tok == e_tok).all(), f"{what}: ids are not the commit rule on the CUDA path's own confidences"
        if g_n is not None:
            assert (np.asarray(g_n) == e_n).all(), f"{what}: counts are not the commit rule's"
    diff = (g_tok != r_tokens) | (_masked_bits(g_mask, S) != _masked_bits(r_mask, S))
    bad = diff & ~r_tie
    assert not bad.any(), f"{what}: CUDA path and oracle differ at non-tie positions {np.argwhere(bad)[:8].tolist()}"
    if g_n is not None and r_n is not None:
        clean = ~r_tie.any(axis=1)
        assert (np.asarray(g_n)[clean] == np.asarray(r_n)[clean]).all(), f"{what}: commit counts differ"
    masked = _masked_bits(mask, S)
    flagged, compared = int((r_tie & masked).sum()), int(masked.sum())
    near_tie_log.record(os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], flagged, compared)
    return flagged, compared


def probe_rows(dec, mask, S):
    """Original rows (b*S + i) in the order the probe reports activations:
    with active-sequence compaction (the default), the rows of the sequences
    that had a masked position before the step, in sequence order."""
    from block_wise_masked_dd_b300.decoder import active_rows
    return active_rows(mask, S, dec.compact_sequences and not dec.fused_reduce)


def with_finished(cfg, tok, mask, finished, seed=0):
    """The state (tok, mask) with the sequences in `finished` fully committed
    (mask word 0, every position holding a seeded id in [0, V))."""
    tok, mask = tok.copy(), mask.copy()
    rng = np.random.default_rng(seed)
    for b in finished:
        tok[b] = rng.integers(0, cfg.vocab, cfg.block, dtype=np.int32)
        mask[b] = 0
    return tok, mask


def compare_step(p: Problem, tok, mask, gamma, mode=0, logits=True):
    """Run one step on both sides from the same state; check every probe.
    Returns (gpu new tokens, gpu new mask, oracle result, near-tie count)."""
    cfg = p.cfg
    t, m = p.gpu_state(tok, mask)
    out = p.dec.probe_step(t, m, gamma, mode, logits=logits)
    torch.cuda.synchronize()
    r = oracle.denoise_step(p.model, tok, mask, gamma, mode, keep_intermediates=True)
    from block_wise_masked_dd_b300.decoder import join_split
    rows = probe_rows(p.dec, mask, cfg.block)
    n = rows.size
    for l in range(cfg.n_layers):
        close(join_split(out["attn_out"][l]).cpu().numpy()[:n], r.attn_out[l][rows], TOL_ATTN,
              f"attention output, layer {l}", rel_rms=1e-3)
    close(join_split(out["hidden"]).cpu().numpy()[:n], r.hidden_final[rows], TOL_LOGIT, "final hidden", rel_rms=1e-3)
    if logits:
        close(out["logits"].cpu().numpy()[:n], r.logits[rows], TOL_LOGIT, "logits")
    g_conf = out["conf"].cpu().numpy()
    close(g_conf[rows], r.conf.reshape(-1)[rows], TOL_CONF, "confidence")
    arg = out["arg"].cpu().numpy()
    mism = (arg[rows] != r.arg.reshape(-1)[rows]) & ~r.logit_tie.reshape(-1)[rows]
    assert not mism.any(), f"argmax differs at rows {rows[np.nonzero(mism)[0][:10]]} whose top-2 logit gap is not a near-tie"
    g_tok = t.cpu().numpy()
    g_mask = m.cpu().numpy().view(np.uint32)
    flagged, _ = check_commit(tok, mask, gamma, mode, cfg.block, r.tokens, r.mask, r.near_tie, g_tok, g_mask,
                              out["n_committed"].cpu().numpy(), r.n_committed, g_conf, arg)
    return g_tok, g_mask, r, flagged
