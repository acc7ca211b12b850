"""The tcgen05 context-attention kernel inside the denoising step (split
activations) at every query-group shape it takes (G query heads per kv head
times S block positions = 64 rows): the stacked form (head and remainder rows
of one M = 128 operand) at G = 2, 4 and 8, and the two-pass M = 64 form at
G = 16, against the oracle, from the start of a block and from a partly
committed state, with a context whose last key tile is ragged; and with
context keys that grow tile by tile, so that the kernels move their
reference maxima (and rescale the accumulated outputs) after the first tile."""
import pytest

import synth
from tests.gpu_helpers import Problem, compare_step, require_gpu

pytestmark = pytest.mark.gpu


def _cfg(batch, block, hq, hkv, ctx=300):
    return synth.Config(f"g{hq // hkv}s{block}", batch=batch, block=block, hidden=512, n_q_heads=hq, n_kv_heads=hkv,
                        head_dim=128, n_layers=2, mlp=1024, vocab=4096, ctx_len=ctx, max_ctx=ctx)


SHAPES = {
    "G2_S32": _cfg(1, 32, 4, 2),
    "G4_S16": _cfg(2, 16, 8, 2),
    "G8_S8": _cfg(2, 8, 8, 1, ctx=777),
    "G16_S4": _cfg(4, 4, 16, 1, ctx=129),
}


@pytest.fixture(scope="module", params=list(SHAPES))
def prob(request):
    require_gpu()
    p = Problem(SHAPES[request.param])
    yield p
    p.dec.close()


def test_first_step(prob):
    tok, mask = prob.start_state()
    compare_step(prob, tok, mask, 0.8)


def test_partly_committed_step(prob):
    tok, mask = synth.make_tokens(prob.cfg, seed=41, masked_frac=0.5)
    compare_step(prob, tok, mask, 0.8, logits=False)


# 64 (sequence, kv head) pairs and 5 context tiles: two context splits of
# up to three tiles, so the reference maxima move inside a work item
GROWING = {"G4_S16": _cfg(32, 16, 8, 2, ctx=640), "G16_S4": _cfg(64, 4, 16, 1, ctx=640)}


@pytest.mark.parametrize("shape", list(GROWING))
def test_first_step_with_growing_keys(shape):
    require_gpu()
    p = Problem(GROWING[shape], seed=3, key_growth=16.0)
    try:
        tok, mask = p.start_state()
        compare_step(p, tok, mask, 0.8)
    finally:
        p.dec.close()
