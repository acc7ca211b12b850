"""The large decode workload on the GPU: batch 32, context 32768, block 16,
hidden 4096, 32 q / 8 kv heads x 128, 8 layers, SwiGLU 14336, vocab 131072,
run at full size in the launch configuration the decoder uses, and checked
against the oracle on sampled sequences (the oracle decodes those sequences
alone: sequences never interact, which the oracle's own batch-independence
pin establishes)."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import TOL_ATTN, TOL_CONF, TOL_LOGIT, check_commit, close, probe_rows, require_gpu, torch

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SAMPLE = [0, 13, 31]


class LargeProblem:
    def __init__(self, sample):
        from block_wise_masked_dd_b300.decoder import Decoder, pack_weights
        cfg = synth.LARGE
        self.cfg = cfg
        self.sample = list(sample)
        w = synth.make_weights_torch(cfg, 0, "cuda")
        k, v = synth.make_context_kv_torch(cfg, 1, "cuda")
        self.dec = Decoder(cfg, pack_weights(cfg, w, "cuda"), "cuda")
        self.dec.set_context_kv(k, v, 0)
        idx = torch.tensor(self.sample, device="cuda")
        k_s = k.index_select(1, idx).float().cpu().numpy()
        v_s = v.index_select(1, idx).float().cpu().numpy()
        del k, v
        wf = {n: t.float().cpu().numpy() for n, t in w.items()}
        del w
        torch.cuda.synchronize()
        sub = dataclasses.replace(cfg, batch=len(self.sample))
        self.model = oracle.OracleModel(sub, wf, k_s, v_s, cfg.ctx_len)

    def rows(self):
        S = self.cfg.block
        return np.concatenate([np.arange(b * S, (b + 1) * S) for b in self.sample])

    def compare(self, tok, mask, gamma, mode=0, logits=True):
        """One step of the whole batch on the GPU from (tok, mask); the sampled
        sequences are checked against the oracle run from the same state."""
        from block_wise_masked_dd_b300.decoder import join_split
        cfg, sel, rows = self.cfg, self.sample, self.rows()
        t = torch.from_numpy(tok.copy()).cuda()
        m = torch.from_numpy(mask.view(np.int32).copy()).cuda()
        out = self.dec.probe_step(t, m, gamma, mode, logits=logits)
        torch.cuda.synchronize()
        r = oracle.denoise_step(self.model, tok[sel], mask[sel], gamma, mode, keep_intermediates=True)
        # probe activations come in the compacted order of the active sequences
        order = {int(row): k for k, row in enumerate(probe_rows(self.dec, mask, cfg.block))}
        act = np.array([row in order for row in rows])
        prow = np.array([order[row] for row in rows[act]], np.int64)
        for l in range(cfg.n_layers):
            got = join_split(out["attn_out"][l]).cpu().numpy()[prow]
            close(got, r.attn_out[l][act], TOL_ATTN, f"attention output, layer {l}", rel_rms=1e-3)
        close(join_split(out["hidden"]).cpu().numpy()[prow], r.hidden_final[act], TOL_LOGIT, "final hidden",
              rel_rms=1e-3)
        if logits:
            close(out["logits"].cpu().numpy()[prow], r.logits[act], TOL_LOGIT, "logits")
        rows = rows[act]
        r_conf, r_arg, r_tie = (r.conf.reshape(-1)[act], r.arg.reshape(-1)[act], r.logit_tie.reshape(-1)[act])
        g_conf = out["conf"].cpu().numpy()
        close(g_conf[rows], r_conf, TOL_CONF, "confidence")
        arg = out["arg"].cpu().numpy()
        mism = (arg[rows] != r_arg) & ~r_tie
        assert not mism.any(), f"argmax differs at non-tie rows {rows[np.nonzero(mism)[0][:10]]}"
        g_tok = t.cpu().numpy()
        g_mask = m.cpu().numpy().view(np.uint32)
        g_n = out["n_committed"].cpu().numpy()
        # the whole batch commits by the rule on its own confidences ...
        e_tok, e_mask, e_n, _ = oracle.commit(g_conf.reshape(cfg.batch, cfg.block), arg.reshape(cfg.batch, cfg.block),
                                              tok, mask, gamma, mode, cfg.block)
        assert (g_tok == e_tok).all() and (g_mask == e_mask).all() and (g_n == e_n).all()
        # ... and the sample differs from the oracle only at its near-ties
        flagged, _ = check_commit(tok[sel], mask[sel], gamma, mode, cfg.block, r.tokens, r.mask, r.near_tie,
                                  g_tok[sel], g_mask[sel], g_n[sel], r.n_committed, what="large step")
        # every sequence (sampled or not) committed at least one masked position
        newly = mask & ~g_mask
        assert ((newly != 0) | (mask == 0)).all()
        assert ((g_mask & ~mask) == 0).all()
        return g_tok, g_mask, flagged


@pytest.fixture(scope="module")
def large():
    require_gpu()
    free, _ = torch.cuda.mem_get_info()
    if free < 100 * 2 ** 30:
        pytest.skip("the large workload needs ~100 GB of free device memory")
    return LargeProblem(SAMPLE)


def start_state(cfg):
    return (np.full((cfg.batch, cfg.block), cfg.vocab, np.int32),
            np.full(cfg.batch, (1 << cfg.block) - 1, np.uint32))


def test_large_state_synced_decode(large):
    """gamma 0.8 through a whole block; every step compared on the sample."""
    tok, mask = start_state(large.cfg)
    steps = ties = 0
    while mask.max():
        tok, mask, t = large.compare(tok, mask, 0.8, logits=(steps == 0))
        ties += t
        steps += 1
        assert steps <= large.cfg.block
    assert (tok < large.cfg.vocab).all()
    print(f"large, gamma 0.8: {steps} steps, {ties} near-tie positions in the sample")


@pytest.mark.parametrize("gamma,mode", [(0.5, 0), (0.95, 0), (0.8, 1)])
def test_large_first_step(large, gamma, mode):
    tok, mask = start_state(large.cfg)
    large.compare(tok, mask, gamma, mode, logits=False)


@pytest.mark.parametrize("gamma,mode", [(0.5, 0), (0.8, 0), (0.95, 0), (0.8, 1)])
def test_large_decode_block_invariants(large, gamma, mode):
    cfg = large.cfg
    tokens, steps = large.dec.decode_block(gamma, mode)
    torch.cuda.synchronize()
    tok = tokens.cpu().numpy()
    assert ((tok >= 0) & (tok < cfg.vocab)).all()
    if mode == 1:
        assert steps == cfg.block
    else:
        assert 1 <= steps <= cfg.block
    large.dec.device_status()


@pytest.mark.parametrize("masked_frac", [0.3, 0.05])
def test_large_graph_step_compacted_lm_head(large, masked_frac):
    """The step graph (LM head over the compacted masked rows: four M tiles,
    the empty ones skipped) against the oracle on the sampled sequences."""
    cfg = large.cfg
    tok, mask = synth.make_tokens(cfg, seed=int(masked_frac * 100) + 7, masked_frac=masked_frac)
    t = torch.from_numpy(tok.copy()).cuda()
    m = torch.from_numpy(mask.view(np.int32).copy()).cuda()
    large.dec.denoise_step(t, m, 0.8, 0)
    torch.cuda.synchronize()
    sel = large.sample
    r = oracle.denoise_step(large.model, tok[sel], mask[sel], 0.8, 0)
    g_tok, g_mask = t.cpu().numpy(), m.cpu().numpy().view(np.uint32)
    check_commit(tok[sel], mask[sel], 0.8, 0, cfg.block, r.tokens, r.mask, r.near_tie, g_tok[sel], g_mask[sel],
                 what="large graph step")


def test_large_graph_step_with_finished_sequences(large):
    """20 of the 32 sequences finished (among them one sampled): 12 active
    sequences = 192 rows, so the linear layers skip their second 256-row
    tile and the attention runs 12 sequences' work items."""
    from tests.gpu_helpers import with_finished
    cfg = large.cfg
    finished = [b for b in range(cfg.batch) if b % 8 not in (0, 3, 7)]
    assert 13 in finished and 0 not in finished and 31 not in finished
    tok, mask = synth.make_tokens(cfg, seed=31, masked_frac=0.5)
    tok, mask = with_finished(cfg, tok, mask, finished)
    t = torch.from_numpy(tok.copy()).cuda()
    m = torch.from_numpy(mask.view(np.int32).copy()).cuda()
    large.dec.denoise_step(t, m, 0.8, 0)
    torch.cuda.synchronize()
    sel = large.sample
    r = oracle.denoise_step(large.model, tok[sel], mask[sel], 0.8, 0)
    g_tok, g_mask = t.cpu().numpy(), m.cpu().numpy().view(np.uint32)
    check_commit(tok[sel], mask[sel], 0.8, 0, cfg.block, r.tokens, r.mask, r.near_tie, g_tok[sel], g_mask[sel],
                 what="large compacted graph step")
    assert (g_tok[finished] == tok[finished]).all() and (g_mask[finished] == 0).all()


def test_large_compacted_and_uncompacted_decode_agree(large):
    results = []
    for compact in (True, False):
        large.dec.compact_sequences = compact
        tokens, steps = large.dec.decode_block(0.8)
        torch.cuda.synchronize()
        results.append((tokens.cpu().numpy(), steps))
    large.dec.compact_sequences = True
    (a, sa), (b, sb) = results
    assert sa == sb and (a == b).all()
