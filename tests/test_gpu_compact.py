"""Active-sequence compaction: a denoising step runs only the rows of the
sequences that still have a masked position (a finished block needs no more
steps, explainer section "拡散言語モデルで推論するには", step 5; sequences never
interact).  Checked against the oracle from states where some sequences have
finished (the probe path and the step graph), and against the uncompacted
step, which must give identical ids: a row's arithmetic does not depend on
where it sits."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import Problem, check_commit, compare_step, require_gpu, torch, with_finished

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny4():
    require_gpu()
    return Problem(synth.TINY.replace(batch=4))


@pytest.fixture(scope="module")
def tiny16():
    require_gpu()
    return Problem(synth.TINY.replace(batch=16))


@pytest.fixture(scope="module")
def small():
    require_gpu()
    return Problem(synth.SMALL)


def _graph_step(p, tok, mask, gamma=0.8, mode=0):
    t, m = p.gpu_state(tok, mask)
    n = torch.empty(p.cfg.batch, dtype=torch.int32, device="cuda")
    p.dec.denoise_step(t, m, gamma, mode, n_committed=n)
    torch.cuda.synchronize()
    return t.cpu().numpy(), m.cpu().numpy().view(np.uint32), n.cpu().numpy()


@pytest.mark.parametrize("finished", [[1, 2], [0], [3], [0, 1, 2]])
@pytest.mark.parametrize("compact", [True, False])
def test_probe_step_with_finished_sequences(tiny4, finished, compact):
    tiny4.dec.compact_sequences = compact
    try:
        tok, mask = synth.make_tokens(tiny4.cfg, seed=21, masked_frac=0.5)
        tok, mask = with_finished(tiny4.cfg, tok, mask, finished)
        g_tok, g_mask, _, _ = compare_step(tiny4, tok, mask, 0.8)
        # finished sequences are left exactly as they were
        for b in finished:
            assert g_mask[b] == 0 and (g_tok[b] == tok[b]).all()
    finally:
        tiny4.dec.compact_sequences = True


@pytest.mark.parametrize("finished", [[1, 3, 4], list(range(7)), [0, 2, 4, 6]])
def test_graph_step_with_finished_sequences_small(small, finished):
    cfg = small.cfg
    tok, mask = synth.make_tokens(cfg, seed=22, masked_frac=0.4)
    tok, mask = with_finished(cfg, tok, mask, finished)
    g_tok, g_mask, n = _graph_step(small, tok, mask)
    r = oracle.denoise_step(small.model, tok, mask, 0.8)
    check_commit(tok, mask, 0.8, 0, cfg.block, r.tokens, r.mask, r.near_tie, g_tok, g_mask, n, r.n_committed,
                 what="compacted graph step")
    assert (n[finished] == 0).all()


@pytest.mark.parametrize("finished", [list(range(0, 16, 2)), list(range(1, 16)), list(range(9))])
def test_graph_step_with_finished_sequences_two_lm_tiles(tiny16, finished):
    """256 rows (the LM head over two row tiles compacts the masked rows as well)."""
    cfg = tiny16.cfg
    tok, mask = synth.make_tokens(cfg, seed=23, masked_frac=0.6)
    tok, mask = with_finished(cfg, tok, mask, finished)
    g_tok, g_mask, n = _graph_step(tiny16, tok, mask)
    r = oracle.denoise_step(tiny16.model, tok, mask, 0.8)
    check_commit(tok, mask, 0.8, 0, cfg.block, r.tokens, r.mask, r.near_tie, g_tok, g_mask, n, r.n_committed,
                 what="compacted graph step, two LM row tiles")


def test_graph_step_with_every_sequence_finished(small):
    """No active sequence: the step changes nothing and reports no timeout."""
    cfg = small.cfg
    tok = np.arange(cfg.batch * cfg.block, dtype=np.int32).reshape(cfg.batch, cfg.block) % cfg.vocab
    mask = np.zeros(cfg.batch, np.uint32)
    g_tok, g_mask, n = _graph_step(small, tok, mask)
    assert (g_tok == tok).all() and (g_mask == 0).all() and (n == 0).all()
    small.dec.device_status()


@pytest.mark.parametrize("prob,gamma,mode", [("small", 0.8, 0), ("small", 0.5, 0), ("tiny16", 0.8, 0),
                                             ("tiny16", 0.95, 0), ("small", 0.8, oracle.with_param(2, 3))])
def test_compacted_and_uncompacted_decode_agree(prob, gamma, mode, request):
    """The device-side decode loop with and without compaction: the same ids
    and the same number of steps (bit-identical arithmetic per row)."""
    p = request.getfixturevalue(prob)
    results = []
    for compact in (True, False):
        p.dec.compact_sequences = compact
        tokens, steps = p.dec.decode_block(gamma, mode)
        torch.cuda.synchronize()
        results.append((tokens.cpu().numpy(), steps))
    p.dec.compact_sequences = True
    (a, sa), (b, sb) = results
    assert sa == sb and (a == b).all()
    p.dec.device_status()
