"""Shared set-up for the GPU parity tests: inputs from `synth`, the CUDA path
through the C-ABI, the expected values from `oracle`."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth

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

    def __init__(self, cfg: synth.Config, seed: int = 0, device="cuda"):
        from block_wise_masked_dd_b300.decoder import Decoder, pack_weights
        self.cfg = cfg
        self.w_bits = synth.make_weights(cfg, seed)
        self.k_bits, self.v_bits = synth.make_context_kv(cfg, seed)
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


def compare_step(p: Problem, tok, mask, gamma, mode=0, logits=True):
    """Run one step on both sides from the same state; check every probe.
    Returns (gpu new tokens, gpu new mask, oracle result, near-tie count)."""
    cfg = p.cfg
    t, m = p.gpu_state(tok, mask)
    out = p.dec.probe_step(t, m, gamma, mode, logits=logits)
    torch.cuda.synchronize()
    r = oracle.denoise_step(p.model, tok, mask, gamma, mode, keep_intermediates=True)
    from block_wise_masked_dd_b300.decoder import join_split
    for l in range(cfg.n_layers):
        close(join_split(out["attn_out"][l]).cpu().numpy(), r.attn_out[l], TOL_ATTN, f"attention output, layer {l}",
              rel_rms=1e-3)
    close(join_split(out["hidden"]).cpu().numpy(), r.hidden_final, TOL_LOGIT, "final hidden", rel_rms=1e-3)
    if logits:
        close(out["logits"].cpu().numpy(), r.logits, TOL_LOGIT, "logits")
    close(out["conf"].cpu().numpy(), r.conf.reshape(-1), TOL_CONF, "confidence")
    tie = r.near_tie.reshape(-1)
    arg = out["arg"].cpu().numpy()
    want = r.arg.reshape(-1)
    mism = (arg != want) & ~tie
    assert not mism.any(), f"argmax differs at non-tie rows {np.nonzero(mism)[0][:10]}"
    g_tok = t.cpu().numpy()
    g_mask = m.cpu().numpy().view(np.uint32)
    # committed sets and ids agree, except in sequences with a flagged position
    for b in range(cfg.batch):
        if tie[b * cfg.block:(b + 1) * cfg.block].any():
            continue
        assert g_mask[b] == r.mask[b], f"seq {b}: mask {g_mask[b]:#x} vs oracle {r.mask[b]:#x}"
        assert (g_tok[b] == r.tokens[b]).all(), f"seq {b}: tokens differ"
        assert out["n_committed"][b].item() == r.n_committed[b]
    return g_tok, g_mask, r, int(tie.sum())
