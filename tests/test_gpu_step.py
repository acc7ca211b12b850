"""Denoising-step and decode-loop parity through the C-ABI against the oracle,
plus the decode invariants, on the tiny and small decode workloads."""
import dataclasses

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import Problem, check_commit, compare_step, require_gpu, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    require_gpu()
    return Problem(synth.TINY)


@pytest.fixture(scope="module")
def small():
    require_gpu()
    return Problem(synth.SMALL)


def test_tiny_first_step(tiny):
    tok, mask = tiny.start_state()
    compare_step(tiny, tok, mask, 0.8)


def test_tiny_partial_state_step(tiny):
    tok, mask = synth.make_tokens(tiny.cfg, seed=3, masked_frac=0.5)
    compare_step(tiny, tok, mask, 0.8)


@pytest.mark.parametrize("gamma,mode", [(0.5, 0), (0.8, 0), (0.95, 0), (0.8, 1)])
def test_tiny_state_synced_decode(tiny, gamma, mode):
    """Step until full; each step compared from the CUDA path's own state."""
    tok, mask = tiny.start_state()
    steps = 0
    while mask.max():
        tok, mask, _, _ = compare_step(tiny, tok, mask, gamma, mode)
        steps += 1
        assert steps <= 16
    assert (tok < tiny.cfg.vocab).all()


def _free_running_vs_oracle(p, gamma=0.8, mode=0):
    """The free-running decode (the device-side loop graph) against the
    oracle's free-running decode.  Where the two trajectories part, the step
    graph replays the CUDA trajectory one step at a time from the same start
    (it must reproduce the loop's result), and the first step at which the
    two states differ must differ only at positions the oracle flags there."""
    cfg = p.cfg
    tokens, steps = p.dec.decode_block(gamma, mode)
    torch.cuda.synchronize()
    want, w_steps, _ = oracle.decode_block(p.model, gamma, mode)
    got = tokens.cpu().numpy()
    if (got == want).all():
        assert steps == w_steps
        return
    tok, mask = p.start_state()
    for step in range(4 * cfg.block):
        t, m = p.gpu_state(tok, mask)
        p.dec.denoise_step(t, m, gamma, mode)
        torch.cuda.synchronize()
        g_tok, g_mask = t.cpu().numpy(), m.cpu().numpy().view(np.uint32)
        r = oracle.denoise_step(p.model, tok, mask, gamma, mode)
        if not ((g_tok == r.tokens).all() and (g_mask == r.mask).all()):
            check_commit(tok, mask, gamma, mode, cfg.block, r.tokens, r.mask, r.near_tie, g_tok, g_mask,
                         what=f"first divergent step {step}")
            assert r.near_tie.any()
            break
        tok, mask = g_tok, g_mask
        assert mask.max(), "the trajectories agreed to the end but the final ids differ"
    # the step-by-step CUDA trajectory reproduces the loop graph's result
    while mask.max():
        t, m = p.gpu_state(tok, mask)
        p.dec.denoise_step(t, m, gamma, mode)
        torch.cuda.synchronize()
        tok, mask = t.cpu().numpy(), m.cpu().numpy().view(np.uint32)
    assert (tok == got).all()


def test_tiny_decode_block_matches_oracle(tiny):
    _free_running_vs_oracle(tiny)


@pytest.mark.parametrize("gamma", [0.5, 0.8])
def test_small_decode_block_matches_oracle(small, gamma):
    """The product path (the loop graph, with active-sequence compaction)
    free-running on the small workload, 8 sequences."""
    _free_running_vs_oracle(small, gamma)


def test_small_first_step(small):
    tok, mask = small.start_state()
    compare_step(small, tok, mask, 0.8)


@pytest.mark.parametrize("gamma", [0.5, 0.8, 0.95])
def test_small_state_synced_decode(small, gamma):
    tok, mask = small.start_state()
    steps = 0
    ties = 0
    while mask.max():
        tok, mask, _, t = compare_step(small, tok, mask, gamma, logits=(steps == 0))
        ties += t
        steps += 1
        assert steps <= 16
    print(f"gamma={gamma}: {steps} steps, {ties} near-tie positions")


# ------------------------------------------------------------- invariants

def test_gamma_zero_fills_in_one_step(tiny):
    _, steps = tiny.dec.decode_block(0.0)
    assert steps == 1


def test_gamma_above_one_takes_block_steps(small):
    tokens, steps = small.dec.decode_block(1.5)
    assert steps == small.cfg.block


def test_mock_ar_left_to_right(tiny):
    cfg = tiny.cfg
    tok, mask = tiny.start_state()
    t, m = tiny.gpu_state(tok, mask)
    for step in range(cfg.block):
        tiny.dec.denoise_step(t, m, 0.8, 1)
        want = (0xFFFF & ~((1 << (step + 1)) - 1))
        assert int(m.cpu().numpy().view(np.uint32)[0]) == want


def test_committed_positions_never_change(small):
    cfg = small.cfg
    tok, mask = small.start_state()
    t, m = small.gpu_state(tok, mask)
    n = torch.empty(cfg.batch, dtype=torch.int32, device="cuda")
    prev_t, prev_m = t.cpu().numpy().copy(), m.cpu().numpy().view(np.uint32).copy()
    while prev_m.max():
        small.dec.denoise_step(t, m, 0.9, 0, n)
        cur_t, cur_m = t.cpu().numpy(), m.cpu().numpy().view(np.uint32)
        for b in range(cfg.batch):
            committed = ~np.array([(int(prev_m[b]) >> i) & 1 for i in range(16)], bool)
            assert (cur_t[b][committed] == prev_t[b][committed]).all()
            assert int(cur_m[b]) & ~int(prev_m[b]) == 0
            if prev_m[b]:
                assert n[b].item() >= 1 and n[b].item() == bin(int(prev_m[b]) & ~int(cur_m[b])).count("1")
        prev_t, prev_m = cur_t.copy(), cur_m.copy()


def test_step_limit_reported(tiny):
    from block_wise_masked_dd_b300 import binding as B
    with pytest.raises(B.DDError) as e:
        tiny.dec.decode_block(1.5, max_steps=3)
    assert e.value.status == B.DD_ERR_STEP_LIMIT


def test_host_buffers_through_the_abi(tiny):
    """dd_decode_block / dd_denoise_step accept host memory for tokens and mask."""
    cfg = tiny.cfg
    d_tok, _ = tiny.dec.decode_block(0.8)
    h_tok = torch.zeros((cfg.batch, cfg.block), dtype=torch.int32).pin_memory()
    _, steps = tiny.dec.decode_block(0.8, tokens=h_tok)
    torch.cuda.synchronize()
    assert (h_tok.numpy() == d_tok.cpu().numpy()).all()


def test_decode_block_runs_the_device_side_loop(small):
    """dd_decode_block repeats the step inside one graph (conditional while
    node) and gives the same block as stepping the single-step graph."""
    from block_wise_masked_dd_b300 import binding as B
    dec = small.dec
    tok, mask = small.start_state()
    t, m = small.gpu_state(tok, mask)
    kinds = B.dd_profile_step(dec.ctx, t.data_ptr(), m.data_ptr(), 0.8, 0,
                              stream=torch.cuda.current_stream().cuda_stream)
    assert B.dd_step_launch_count(dec.ctx) == len(kinds) + 1   # + the loop-control kernel
    tokens, steps = dec.decode_block(0.8)
    torch.cuda.synchronize()
    t, m = small.gpu_state(tok, mask)
    n = 0
    while int(m.max().item()) != 0:
        dec.denoise_step(t, m, 0.8)
        n += 1
    torch.cuda.synchronize()
    assert n == steps
    assert (t.cpu().numpy() == tokens.cpu().numpy()).all()


@pytest.mark.parametrize("mode", [oracle.with_param(oracle.MODE_TOPK, 3), oracle.with_param(oracle.MODE_STEPS, 5)])
def test_tiny_state_synced_topk_and_fixed_steps(tiny, mode):
    tok, mask = tiny.start_state()
    steps = 0
    while mask.max():
        tok, mask, _, _ = compare_step(tiny, tok, mask, 0.8, mode)
        steps += 1
        assert steps <= 16
    assert steps == (6 if (mode & 0xFF) == oracle.MODE_TOPK else 5)


@pytest.mark.parametrize("N", [1, 4, 16])
def test_decode_block_fixed_steps(small, N):
    _, steps = small.dec.decode_block(0.8, oracle.with_param(oracle.MODE_STEPS, N))
    assert steps == N


# ------------------------------------------------------------------- RoPE

@pytest.fixture(scope="module")
def tiny_rope():
    require_gpu()
    return Problem(synth.TINY.replace(rope_theta=10000.0))


@pytest.mark.parametrize("gamma,mode", [(0.8, 0), (0.8, 1)])
def test_tiny_rope_state_synced_decode(tiny_rope, gamma, mode):
    tok, mask = tiny_rope.start_state()
    steps = 0
    while mask.max():
        tok, mask, _, _ = compare_step(tiny_rope, tok, mask, gamma, mode)
        steps += 1
        assert steps <= 16


def test_small_rope_first_step():
    require_gpu()
    p = Problem(synth.SMALL.replace(rope_theta=10000.0))
    tok, mask = p.start_state()
    compare_step(p, tok, mask, 0.8)
    tok, mask = synth.make_tokens(p.cfg, seed=9, masked_frac=0.4)
    compare_step(p, tok, mask, 0.8)


# ------------------------------------------------------ context tower on device

@pytest.mark.parametrize("cfg", [synth.TINY.replace(max_ctx=256 + 32), synth.SMALL],
                         ids=["tiny", "small"])
def test_append_block_then_next_block_matches_oracle(cfg):
    """Decode a block, encode it with the context tower on the device, then step
    the next block state-synced against the oracle's own append (twice)."""
    require_gpu()
    p = Problem(cfg)
    tw_bits = synth.make_tower_weights(cfg, 0)
    tw = {k: synth.bf16_bits_to_f32(v) for k, v in tw_bits.items()}
    p.dec.set_context_tower(tw_bits)
    for blk in range(2):
        tokens, _ = p.dec.decode_block(0.8)
        p.dec.append_block(tokens)
        torch.cuda.synchronize()
        p.model = oracle.append_block(p.model, tw, tokens.cpu().numpy())
        tok, mask = p.start_state()
        steps = 0
        while mask.max() and steps < (16 if cfg.name == "tiny" else 3):
            tok, mask, _, _ = compare_step(p, tok, mask, 0.8, logits=(steps == 0))
            steps += 1


# --------------------------------------------------------- empty context

@pytest.mark.parametrize("which", ["tiny", "small"])
def test_step_with_empty_context(which, request):
    """Context length 0: each query attends to the block keys alone (every
    context split of the tcgen05 path, and the mma.sync path's context loop,
    is empty)."""
    import copy
    p = request.getfixturevalue(which)
    q = copy.copy(p)
    q.model = dataclasses.replace(p.model, ctx_len=0)
    p.dec.set_context_len(0)
    try:
        tok, mask = q.start_state()
        compare_step(q, tok, mask, 0.8)
        tok, mask = synth.make_tokens(q.cfg, seed=21, masked_frac=0.5)
        compare_step(q, tok, mask, 0.8, logits=False)
    finally:
        p.dec.set_context_len(p.cfg.ctx_len)


# ------------------------------------------- LM head over the compacted rows

def _graph_step_vs_oracle(p, tok, mask, gamma=0.8):
    """One step through the step graph (LM head over the compacted masked rows)
    against the oracle: they may differ only at the oracle's near-ties."""
    cfg = p.cfg
    t, m = p.gpu_state(tok, mask)
    n = torch.empty(cfg.batch, dtype=torch.int32, device="cuda")
    p.dec.denoise_step(t, m, gamma, 0, n_committed=n)
    torch.cuda.synchronize()
    r = oracle.denoise_step(p.model, tok, mask, gamma, 0)
    g_tok, g_mask = t.cpu().numpy(), m.cpu().numpy().view(np.uint32)
    check_commit(tok, mask, gamma, 0, cfg.block, r.tokens, r.mask, r.near_tie, g_tok, g_mask, n.cpu().numpy(),
                 r.n_committed, what="graph step")


@pytest.mark.parametrize("masked_frac", [1.0, 0.6, 0.3, 0.05])
def test_compacted_lm_head_two_row_tiles(masked_frac):
    """256 rows (two M tiles of the LM head): masked-row counts above 128,
    between 64 and 128 and at most 64 (a CTA whose only tile has no row left
    still runs it, with its outputs dropped)."""
    require_gpu()
    p = Problem(synth.TINY.replace(batch=16))
    if masked_frac == 1.0:
        tok, mask = p.start_state()
    else:
        tok, mask = synth.make_tokens(p.cfg, seed=int(masked_frac * 100), masked_frac=masked_frac)
    _graph_step_vs_oracle(p, tok, mask)


@pytest.mark.parametrize("masked_frac", [0.6, 0.3, 0.05])
def test_compacted_lm_head_small(small, masked_frac):
    """128 rows, one M tile: the step graph with partly filled blocks (no
    compaction, since the single tile always runs)."""
    tok, mask = synth.make_tokens(small.cfg, seed=int(masked_frac * 100) + 1, masked_frac=masked_frac)
    _graph_step_vs_oracle(small, tok, mask)


def test_weights_set_again_reach_both_graphs():
    """dd_init_weights with another weight set after both graphs were captured:
    the single-step graph and the decode-loop graph then run the new weights,
    bit for bit as a context created with them (the previous weights stay
    allocated meanwhile)."""
    require_gpu()
    from block_wise_masked_dd_b300.decoder import Decoder, pack_weights
    cfg = synth.TINY
    a = Problem(cfg, seed=0)
    w_b = pack_weights(cfg, synth.make_weights(cfg, 1), "cuda")
    fresh = Decoder(cfg, w_b, "cuda")
    fresh.set_context_kv(a.k_dev, a.v_dev, 0)
    ref_block, ref_steps = fresh.decode_block(0.8)
    tok, mask = a.start_state()
    t_ref, m_ref = a.gpu_state(tok, mask)
    fresh.denoise_step(t_ref, m_ref, 0.8)
    old_block, _ = a.dec.decode_block(0.8)  # captures both graphs with the first weights
    t0, m0 = a.gpu_state(tok, mask)
    a.dec.denoise_step(t0, m0, 0.8)
    keep = a.dec.weights
    a.dec.set_weights(w_b)
    new_block, new_steps = a.dec.decode_block(0.8)
    t1, m1 = a.gpu_state(tok, mask)
    a.dec.denoise_step(t1, m1, 0.8)
    torch.cuda.synchronize()
    assert new_steps == ref_steps and torch.equal(new_block, ref_block)
    assert torch.equal(t1, t_ref) and torch.equal(m1, m_ref)
    assert not torch.equal(old_block, new_block)  # the two weight sets decode differently
    fresh.close()
    a.dec.close()
    del keep
