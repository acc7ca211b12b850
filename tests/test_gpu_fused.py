"""The linear layers with the split-K reduction inside the GEMM (groups of CTAs
exchanging partial tiles through L2, deferred RMSNorm) and
the path with separate reduce kernels: both against the oracle, and against
each other, on several row counts (one and several TMEM column blocks, group
sizes from the planner), with and without rotary positions."""
import numpy as np
import pytest

import synth
from tests.gpu_helpers import TOL_CONF, TOL_LOGIT, Problem, close, compare_step, require_gpu, torch

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": synth.TINY,
    "tiny_b3": synth.TINY.replace(batch=3),      # 48 rows: one 16-column TMEM tail only
    "tiny_b5": synth.TINY.replace(batch=5),      # 80 rows: a 64-column block plus a 16-column tail
    "tiny_rope": synth.TINY.replace(rope_theta=10000.0),
    "small": synth.SMALL,
}


@pytest.fixture(scope="module", params=list(CASES))
def prob(request):
    require_gpu()
    p = Problem(CASES[request.param])
    yield p
    p.dec.close()


def test_fused_path_is_planned_and_off_by_default(prob):
    dec = prob.dec
    assert not dec.fused_reduce
    plan = dec.fused_plan()
    print(prob.cfg.batch * prob.cfg.block, "rows:", plan)
    for layer, (cs, grid) in plan.items():
        assert 1 <= cs <= 8, layer
        assert grid >= cs and grid % cs == 0, layer


@pytest.mark.parametrize("fused", [True, False])
def test_both_paths_match_the_oracle(prob, fused):
    prob.dec.fused_reduce = fused
    try:
        tok, mask = prob.start_state()
        compare_step(prob, tok, mask, 0.8)
        tok, mask = synth.make_tokens(prob.cfg, seed=11, masked_frac=0.4)
        compare_step(prob, tok, mask, 0.8, logits=False)
    finally:
        prob.dec.fused_reduce = False


def test_fused_and_separate_reduce_agree(prob):
    """The two paths differ only in rounding order: logits and confidences
    agree far inside the oracle tolerance."""
    tok, mask = synth.make_tokens(prob.cfg, seed=5, masked_frac=0.7)
    outs = []
    for fused in (True, False):
        prob.dec.fused_reduce = fused
        t, m = prob.gpu_state(tok, mask)
        outs.append(prob.dec.probe_step(t, m, 0.8, 0, logits=True))
        torch.cuda.synchronize()
    prob.dec.fused_reduce = False
    a, b = outs
    close(a["logits"].cpu().numpy(), b["logits"].cpu().numpy(), TOL_LOGIT / 4, "logits, fused vs separate")
    close(a["conf"].cpu().numpy(), b["conf"].cpu().numpy(), TOL_CONF / 4, "confidence, fused vs separate")


def test_fused_decode_block_runs_clean(prob):
    """The device-side decode loop over the fused graph: every position is
    committed, ids are in range and no bounded wait expired."""
    prob.dec.fused_reduce = True
    try:
        tokens, steps = prob.dec.decode_block(0.8)
        torch.cuda.synchronize()
    finally:
        prob.dec.fused_reduce = False
    tok = tokens.cpu().numpy()
    assert 1 <= steps <= prob.cfg.block
    assert ((tok >= 0) & (tok < prob.cfg.vocab)).all()
    prob.dec.device_status()


def test_option_errors():
    require_gpu()
    from block_wise_masked_dd_b300 import binding as B
    p = Problem(synth.TINY)
    with pytest.raises(B.DDError):
        B.dd_set_option(p.dec.ctx, B.DD_OPT_FUSED_REDUCE, 2)
    with pytest.raises(B.DDError):
        B.dd_set_option(p.dec.ctx, 77, 1)
    with pytest.raises(B.DDError):
        B.dd_get_option(p.dec.ctx, 77)
    with pytest.raises(B.DDError):
        B.dd_set_option(p.dec.ctx, B.DD_OPT_FUSED_SPLITS["qkv"], 4)
    assert B.dd_get_option(p.dec.ctx, B.DD_OPT_COMPACT_SEQUENCES) == 1     # on by default
    with pytest.raises(B.DDError):
        B.dd_set_option(p.dec.ctx, B.DD_OPT_COMPACT_SEQUENCES, 2)
    B.dd_set_option(p.dec.ctx, B.DD_OPT_COMPACT_SEQUENCES, 0)
    assert B.dd_get_option(p.dec.ctx, B.DD_OPT_COMPACT_SEQUENCES) == 0
    p.dec.close()


def test_unavailable_for_more_than_128_rows():
    """256 rows: the fused path is not planned; asking for it is refused and
    the separate-reduce path runs (and matches the oracle)."""
    require_gpu()
    from block_wise_masked_dd_b300 import binding as B
    p = Problem(synth.TINY.replace(batch=16))
    assert not p.dec.fused_reduce
    assert all(v == (0, 0) for v in p.dec.fused_plan().values())
    with pytest.raises(B.DDError):
        p.dec.fused_reduce = True
    tok, mask = p.start_state()
    compare_step(p, tok, mask, 0.8, logits=False)
    p.dec.close()
