"""The oracle's pins must catch plausible mistakes.

Each mutant below edits the source of one oracle function (a dropped term, a
wrong index or sign, a transposed operand, an off-by-one in the commit rule),
runs on the CPU only, and must make at least one pin of
tests/test_oracle_pins.py fail.  Nothing here touches the CUDA path.
"""
import inspect
import textwrap

import numpy as np
import pytest

import oracle
import oracle.decode as od
import synth
from tests import test_golden
from tests import test_oracle_pins as pins
from tests.golden_io import commit_cases, near_tie_cases

# (function, [(old source text, new source text), ...])
MUTANTS = {
    "attention_without_scale": ("block_attention", [(") * scale", ")")]),
    "attention_gqa_modulo": ("block_attention", [("kvh = h // G", "kvh = h % Hkv")]),
    "attention_drops_context": ("block_attention", [
        ("np.concatenate([k_ctx[kvh], k_blk[:, kvh, :]], axis=0)", "k_blk[:, kvh, :]"),
        ("np.concatenate([v_ctx[kvh], v_blk[:, kvh, :]], axis=0)", "v_blk[:, kvh, :]")]),
    "attention_drops_block": ("block_attention", [
        ("np.concatenate([k_ctx[kvh], k_blk[:, kvh, :]], axis=0)", "np.concatenate([k_ctx[kvh], k_blk[:1, kvh, :]], axis=0)"),
        ("np.concatenate([v_ctx[kvh], v_blk[:, kvh, :]], axis=0)", "np.concatenate([v_ctx[kvh], v_blk[:1, kvh, :]], axis=0)")]),
    "attention_normalises_wrong_axis": ("block_attention", [("p.sum(axis=1,", "p.sum(axis=0,")]),
    "rmsnorm_mean_abs": ("rmsnorm", [("np.mean(x * x,", "np.mean(np.abs(x),")]),
    "rmsnorm_without_gain": ("rmsnorm", [(") * g.astype(F32)", ")")]),
    "rmsnorm_without_eps": ("rmsnorm", [("ms + F32(eps)", "ms")]),
    "silu_is_sigmoid": ("silu", [("return x / (F32(1.0)", "return F32(1.0) / (F32(1.0)")]),
    "argmax_last_on_ties": ("select_from_logits", [
        ("np.argmax(logits, axis=1)", "(logits.shape[1] - 1 - np.argmax(logits[:, ::-1], axis=1))")]),
    "confidence_at_temperature_2": ("select_from_logits", [("np.exp(logits - m)", "np.exp((logits - m) / F32(2.0))")]),
    "round_bf16_ties_away": ("round_bf16", [("np.uint64(0x7FFF) + lsb", "np.uint64(0x8000)")]),
    "commit_strict_threshold": ("commit", [(">= g]", "> g]")]),
    "fallback_last_on_ties": ("commit", [("if F32(conf[b, i]) > F32(conf[b, best]):",
                                          "if F32(conf[b, i]) >= F32(conf[b, best]):")]),
    "mock_ar_rightmost": ("commit", [("chosen = [masked[0]]", "chosen = [masked[-1]]")]),
    "step_drops_attention_residual": ("denoise_step", [("x = x + o @", "x = o @")]),
    "step_swaps_gate_and_up": ("denoise_step", [('silu(y @ w[f"wg{l}"].T) * (y @ w[f"wu{l}"].T)',
                                                 'silu(y @ w[f"wu{l}"].T) * (y @ w[f"wg{l}"].T)')]),
    "step_mask_reads_token_zero": ("denoise_step", [("[[V if (int(mask[b]) >> i) & 1", "[[0 if (int(mask[b]) >> i) & 1")]),
    "step_without_positions": ("denoise_step", [(' + w["pos"][None, :, :]', "")]),
    "step_transposed_wq": ("denoise_step", [('y @ w[f"wq{l}"].T', 'y @ w[f"wq{l}"]')]),
    "step_mlp_norm_gain_from_attention": ("denoise_step", [('w[f"g_mlp{l}"]', 'w[f"g_attn{l}"]')]),
    "topk_ties_to_higher_position": ("commit", [("key=lambda i: (-float(F32(conf[b, i])), i)",
                                                 "key=lambda i: (-float(F32(conf[b, i])), -i)")]),
    "topk_takes_one_more": ("commit", [("chosen = sorted(ranked[:k])", "chosen = sorted(ranked[:k + 1])")]),
    "rope_wrong_sign": ("rope", [("x[..., 0::2] * s + x[..., 1::2] * c", "x[..., 1::2] * c - x[..., 0::2] * s")]),
    "rope_wrong_frequency": ("rope", [("-2.0 * np.arange(D // 2, dtype=np.float64) / D", "-1.0 * np.arange(D // 2, dtype=np.float64) / D")]),
    "step_rope_keys_unrotated": ("denoise_step", [("k = np.stack([rope(k[b], pos, cfg.rope_theta) for b in range(B)])", "pass")]),
    "append_swaps_k_and_v": ("append_block", [("k_new[l] = kv[:, :Hkv * D]", "k_new[l] = kv[:, Hkv * D:]")]),
    "append_without_norm": ("append_block", [('y = rmsnorm(e, tower["ctx_g"], cfg.rms_eps)', 'y = e')]),
    "append_without_residual": ("append_block", [("h = e + linear(", "h = linear(")]),
    "append_second_norm_uses_first_gain": ("append_block", [('tower["ctx_g2"]', 'tower["ctx_g"]')]),
    "append_attends_without_positions_order": ("append_block", [
        ("a = np.stack([tower_causal_attention(qkv[b, :, 0], qkv[b, :, 1], qkv[b, :, 2]) for b in range(B)])",
         "a = np.stack([tower_causal_attention(qkv[b, :, 0], qkv[b, :, 2], qkv[b, :, 1]) for b in range(B)])")]),
    "tower_attention_not_causal": ("tower_causal_attention", [("s = np.where(np.tril(np.ones((S, S), bool)), s, F32(-np.inf))", "pass")]),
    "tower_attention_without_scale": ("tower_causal_attention", [(") * scale", ")")]),
    "tower_attention_anticausal": ("tower_causal_attention", [("np.tril(np.ones((S, S), bool))", "np.triu(np.ones((S, S), bool))")]),
    "steps_schedule_off_by_one": ("steps_schedule_k", [("steps_left = n_steps - t\n", "steps_left = n_steps - t + 1\n")]),
    # near-tie flags: thresholds, the pairs compared, the modes and positions they cover
    "tie_logit_gap_doubled": ("near_tie_positions", [("if gap[b, i] < TIE_LOGIT_GAP:", "if gap[b, i] < 2 * TIE_LOGIT_GAP:")]),
    "tie_gap_top1_minus_top3": ("top2_gap", [("-np.partition(-logits, 1, axis=1)[:, :2]",
                                               "-np.partition(-logits, 2, axis=1)[:, [0, 2]]")]),
    "tie_flags_every_masked": ("near_tie_positions", [("if gap[b, i] < TIE_LOGIT_GAP:", "if True:")]),
    "tie_gamma_ignored": ("near_tie_positions", [("if abs(conf[b, i] - gamma) < TIE_GAMMA_GAP:", "if False:")]),
    "tie_gamma_gap_tenfold": ("near_tie_positions", [("if abs(conf[b, i] - gamma) < TIE_GAMMA_GAP:",
                                                      "if abs(conf[b, i] - gamma) < 10 * TIE_GAMMA_GAP:")]),
    "tie_gamma_in_every_mode": ("near_tie_positions", [("if base == MODE_THRESHOLD:",
                                                        "if base in (MODE_THRESHOLD, MODE_MOCK_AR, MODE_TOPK, MODE_STEPS):")]),
    "tie_fallback_wrong_pair": ("near_tie_positions", [("c[0] - c[1] < TIE_CONF_GAP", "c[0] - c[min(2, len(c) - 1)] < TIE_CONF_GAP")]),
    "tie_fallback_missing": ("near_tie_positions", [("if fallback and len(c) > 1", "if False and len(c) > 1")]),
    "tie_fallback_without_fallback": ("near_tie_positions", [("if fallback and len(c) > 1", "if len(c) > 1")]),
    "tie_ranks_committed_positions": ("near_tie_positions", [("c = sorted((conf[b, i] for i in masked), reverse=True)",
                                                              "c = sorted((conf[b, i] for i in range(S)), reverse=True)")]),
    "tie_cut_off_by_one": ("near_tie_positions", [("if 0 < k < len(c) and c[k - 1] - c[k] < TIE_CONF_GAP:",
                                                   "if 0 < k < len(c) - 1 and c[k] - c[k + 1] < TIE_CONF_GAP:")]),
    "tie_cut_missing": ("near_tie_positions", [("if 0 < k < len(c) and c[k - 1] - c[k] < TIE_CONF_GAP:", "if False:")]),
    "tie_steps_wrong_k": ("near_tie_positions", [("else steps_schedule_k(S, param, len(masked))", "else param")]),
    "tie_flags_committed_positions": ("near_tie_positions", [("masked = [i for i in range(S) if (int(mask[b]) >> i) & 1]",
                                                              "masked = list(range(S))")]),
}


def _mutant(fn_name, edits):
    src = textwrap.dedent(inspect.getsource(getattr(od, fn_name)))
    for old, new in edits:
        assert old in src, f"{fn_name}: {old!r} not found"
        src = src.replace(old, new)
    ns = dict(od.__dict__)
    exec(compile(src, f"<mutant of {fn_name}>", "exec"), ns)
    return ns[fn_name]


@pytest.fixture(scope="module")
def tiny_model():
    cfg = synth.TINY.replace(batch=2, ctx_len=64, max_ctx=64)
    return oracle.OracleModel.from_bits(cfg, synth.make_weights(cfg, 0), *synth.make_context_kv(cfg, 0),
                                        synth.bf16_bits_to_f32)


def _pins(tiny):
    """The pins, cheapest first."""
    return [
        pins.test_silu_values,
        pins.test_rmsnorm_closed_forms,
        pins.test_round_bf16_matches_bruteforce,
        pins.test_select_equal_logits,
        lambda: pins.test_select_single_lead_closed_form(3.0),
        pins.test_select_vs_bruteforce_and_first_max,
        lambda: pins.test_attention_vs_bruteforce(17, 4, 1),
        lambda: pins.test_attention_vs_bruteforce(1, 4, 2),
        pins.test_attention_constant_values,
        pins.test_attention_zero_query_is_uniform_mean,
        pins.test_attention_gqa_equals_repeated_mha,
        pins.test_attention_is_bidirectional_and_sees_context,
        pins.test_commit_exhaustive_masks,
        pins.test_commit_gamma_zero_and_above_one,
        pins.test_commit_monotone_in_gamma,
        _golden_commit_cases,
        _golden_near_tie_cases,
        *[lambda g=g, m=m: pins.test_near_tie_flags_are_sound(g, m) for g, m in pins.NEAR_TIE_MODES],
        lambda: pins.test_steps_schedule_fills_block_in_n_steps(16),
        pins.test_commit_topk_exhaustive_masks,
        lambda: pins.test_full_step_vs_bruteforce(False),
        pins.test_full_step_vs_bruteforce_random_gains,
        lambda: pins.test_decode_mock_ar_is_left_to_right(tiny),
        lambda: pins.test_decode_committed_never_change_and_progress(tiny),
        lambda: pins.test_decode_topk_and_fixed_steps(tiny),
        pins.test_rope_closed_forms,
        pins.test_rope_scores_depend_on_relative_position,
        pins.test_full_step_with_rope_vs_bruteforce,
        pins.test_append_block_vs_bruteforce,
        pins.test_append_block_is_causal,
        pins.test_tower_attention_closed_forms,
        lambda: pins.test_decode_after_append_sees_the_new_context(tiny),
    ]


def _golden_near_tie_cases():
    for case in near_tie_cases():
        test_golden.test_near_tie_cases(case)


def _golden_commit_cases():
    for case in commit_cases():
        test_golden.test_commit_rule_cases(case)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch, tiny_model):
    fn_name, edits = MUTANTS[name]
    bad = _mutant(fn_name, edits)
    monkeypatch.setattr(od, fn_name, bad)
    if hasattr(oracle, fn_name):
        monkeypatch.setattr(oracle, fn_name, bad)
    for pin in _pins(tiny_model):
        try:
            with np.errstate(all="ignore"):
                pin()
        except Exception:  # an assertion, or the mutant breaking outright
            return
    pytest.fail(f"no pin caught the mutant {name}")
