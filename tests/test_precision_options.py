"""Why every activation operand of the CUDA path is a bf16 head plus a bf16
remainder: each cheaper option, applied alone at one point of the step (or
one fp16 pass at every GEMM input) and
measured with the oracle on the small decode workload (two sequences, four
layers, a partly committed block), moves some logit past the parity bar
(|d| <= 2e-2 + 2e-2 |logit|).  The variants are the oracle with one operand
rounded to bf16 before its product, built by editing a copy of its source
(the oracle itself is unchanged); the reference is the oracle as it stands.
These measurements fix the design; they pin nothing in the oracle."""
import inspect
import textwrap

import numpy as np
import pytest

import oracle
import oracle.decode as od
import synth

pytestmark = pytest.mark.slow

CFG = synth.SMALL.replace(batch=2)

# point -> edits of oracle.decode source (function, old text, new text)
VARIANTS = {
    "gate|up input": [("denoise_step", 'hmid = st(silu(y @ w[f"wg{l}"].T) * (y @ w[f"wu{l}"].T))',
                       'yb = round_bf16(y)\n        hmid = st(silu(yb @ w[f"wg{l}"].T) * (yb @ w[f"wu{l}"].T))')],
    "down input": [("denoise_step", 'x = x + hmid @ w[f"wd{l}"].T', 'x = x + round_bf16(hmid) @ w[f"wd{l}"].T')],
    "LM-head input": [("denoise_step", 'conf, arg, logits = lm_head_select(hf, w["lm_head"])',
                       'conf, arg, logits = lm_head_select(round_bf16(hf), w["lm_head"])')],
    "attention query": [("block_attention", 's = (q[:, h, :].astype(F32) @ keys.T) * scale',
                         's = (round_bf16(q[:, h, :].astype(F32)) @ keys.T) * scale')],
    "attention probabilities": [("block_attention", "out[:, h, :] = p @ vals", "out[:, h, :] = round_bf16(p) @ vals")],
    # every GEMM input (the four projections and the LM head) rounded once to
    # fp16 (11-bit significand): the weights convert to fp16 exactly in the
    # normal range, so this is a single fp16 tensor-core pass per GEMM
    "every GEMM input in fp16": [("denoise_step", a, b) for a, b in [
        ('q = (y @ w[f"wq{l}"].T)', 'q = (round_fp16(y) @ w[f"wq{l}"].T)'),
        ('k = (y @ w[f"wk{l}"].T)', 'k = (round_fp16(y) @ w[f"wk{l}"].T)'),
        ('v = st(y @ w[f"wv{l}"].T)', 'v = st(round_fp16(y) @ w[f"wv{l}"].T)'),
        ('x = x + o @ w[f"wo{l}"].T', 'x = x + round_fp16(o) @ w[f"wo{l}"].T'),
        ('hmid = st(silu(y @ w[f"wg{l}"].T) * (y @ w[f"wu{l}"].T))',
         'hmid = st(silu(round_fp16(y) @ w[f"wg{l}"].T) * (round_fp16(y) @ w[f"wu{l}"].T))'),
        ('x = x + hmid @ w[f"wd{l}"].T', 'x = x + round_fp16(hmid) @ w[f"wd{l}"].T'),
        ('conf, arg, logits = lm_head_select(hf, w["lm_head"])',
         'conf, arg, logits = lm_head_select(round_fp16(hf), w["lm_head"])')]],
}


def round_fp16(a):
    """fp32 -> nearest fp16 -> fp32 (NumPy's conversion: round to nearest even)."""
    return np.asarray(a, np.float32).astype(np.float16).astype(np.float32)


@pytest.fixture(scope="module")
def problem():
    wb = synth.make_weights(CFG, 0)
    kb, vb = synth.make_context_kv(CFG, 0)
    m = oracle.OracleModel.from_bits(CFG, wb, kb, vb, synth.bf16_bits_to_f32)
    tok, mask = synth.make_tokens(CFG, seed=3, masked_frac=0.6)
    ref = oracle.denoise_step(m, tok, mask, 0.8, keep_intermediates=True)
    return m, tok, mask, ref


def _variant(edits):
    """A namespace holding the edited functions and a denoise_step that calls them."""
    ns = dict(od.__dict__)
    ns["round_fp16"] = round_fp16
    edited = {fn for fn, _, _ in edits}
    for fn in sorted(edited | {"denoise_step"}):
        src = textwrap.dedent(inspect.getsource(getattr(od, fn)))
        for f2, old, new in edits:
            if f2 == fn:
                assert old in src, (fn, old)
                src = src.replace(old, new)
        exec(compile(src, f"<variant of {fn}>", "exec"), ns)
    return ns


@pytest.mark.parametrize("point", sorted(VARIANTS))
def test_single_bf16_operand_breaks_the_logit_bar(problem, point):
    m, tok, mask, ref = problem
    ns = _variant(VARIANTS[point])
    r = ns["denoise_step"](m, tok, mask, 0.8, keep_intermediates=True)
    d = np.abs(r.logits - ref.logits)
    worst = float(np.max(d / (2e-2 + 2e-2 * np.abs(ref.logits))))
    print(f"{point}: max |d logit| {d.max():.3f}, rms {np.sqrt(np.mean(d ** 2)):.4f}, worst / bound {worst:.2f}")
    assert worst > 1.0
