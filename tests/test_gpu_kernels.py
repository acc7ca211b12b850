"""Single-kernel parity through the C-ABI: tensor-core GEMM, block attention,
LM head + confidence select, commit rule, bounded-wait timeout."""
import numpy as np
import pytest

import oracle
import synth
from tests.gpu_helpers import TOL_ATTN, TOL_CONF, bf16_to_f32, close, require_gpu, to_dev, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


# ------------------------------------------------------------------- GEMM

@pytest.mark.parametrize("rows,n,k", [(16, 768, 256), (48, 384, 192), (128, 3072, 2048), (128, 2048, 5632),
                                      (512, 1024, 1024), (272, 256, 640),
                                      (272, 5632, 4096),
                                      # stream-K schedules (tiles cut between CTAs, a slot per piece):
                                      (384, 7168, 4096), (512, 4096, 14336),
                                      # K blocks of 32 without CTA pairs (three weight tiles; an N
                                      # tile of 144 rows), and pairs with 80-row halves (N tile 160)
                                      (272, 384, 1024), (144, 512, 512), (160, 512, 512)])
def test_gemm_vs_oracle_linear(rows, n, k):
    from block_wise_masked_dd_b300.decoder import gemm
    x = synth.make_activations(rows, k, seed=rows + n)
    w = synth.make_activations(n, k, seed=k + 7, std=0.05)
    y = gemm(to_dev(x), to_dev(w))
    torch.cuda.synchronize()
    want = oracle.linear(synth.bf16_bits_to_f32(x), synth.bf16_bits_to_f32(w))
    close(y.cpu().numpy(), want, 1e-3, f"gemm {rows}x{n}x{k}")


# -------------------------------------------------------------- attention

def _attn_case(B, S, Hq, Hkv, D, T, stride, seed, nan_tail=False, key_growth=0.0):
    from block_wise_masked_dd_b300.decoder import block_attention
    qkvw = (Hq + 2 * Hkv) * D
    qkv = synth.make_activations(B * S, qkvw, seed=seed)
    rng = np.random.default_rng(seed + 1)
    k = rng.standard_normal((B, Hkv, stride, D), dtype=np.float32)
    if key_growth:  # keys of 128-position tile t scaled by 1 + key_growth * t
        k *= (1.0 + key_growth * (np.arange(stride) // 128))[:, None].astype(np.float32)
    kc = synth.to_bf16_bits(k)
    vc = synth.to_bf16_bits(rng.standard_normal((B, Hkv, stride, D), dtype=np.float32))
    if nan_tail:  # rows beyond the context length must never reach the output
        kc[:, :, T:, :] = 0x7FC0
        vc[:, :, T:, :] = 0x7FC0
    out = block_attention(to_dev(qkv), to_dev(kc), to_dev(vc), T, B, S, Hq, Hkv, D)
    torch.cuda.synchronize()
    q32 = synth.bf16_bits_to_f32(qkv).reshape(B, S, -1)
    kc32, vc32 = synth.bf16_bits_to_f32(kc), synth.bf16_bits_to_f32(vc)
    got = bf16_to_f32(out).reshape(B, S, Hq, D)
    for b in range(B):
        q = q32[b, :, :Hq * D].reshape(S, Hq, D)
        kb = q32[b, :, Hq * D:(Hq + Hkv) * D].reshape(S, Hkv, D)
        vb = q32[b, :, (Hq + Hkv) * D:].reshape(S, Hkv, D)
        want = oracle.block_attention(q, kb, vb, kc32[b, :, :T], vc32[b, :, :T])
        close(got[b], want, TOL_ATTN, f"attention b={b} T={T}", rel_rms=3e-3)


@pytest.mark.parametrize("B,S,Hq,Hkv,D,T,stride", [
    (2, 16, 8, 2, 128, 200, 256),     # tcgen05 path, NaN rows in the last tile and beyond
    (3, 16, 4, 1, 64, 200, 256),      # mma.sync path
])
def test_block_attention_ignores_rows_beyond_context(B, S, Hq, Hkv, D, T, stride):
    _attn_case(B, S, Hq, Hkv, D, T, stride, seed=5, nan_tail=True)


@pytest.mark.parametrize("B,S,Hq,Hkv,D,T,stride", [
    (1, 16, 4, 4, 64, 256, 256),      # tiny workload shape
    (2, 16, 4, 1, 128, 0, 64),        # no context: block keys only
    (2, 16, 8, 2, 128, 1, 64),        # one context key
    (3, 16, 4, 1, 64, 200, 256),      # ragged last tile, stale rows beyond T
    (2, 8, 8, 1, 128, 777, 800),      # S=8, G=8
    (1, 32, 4, 1, 128, 100, 128),     # S=32: 128 query rows per kv head
    (8, 16, 16, 4, 128, 2048, 2176),  # small decode workload shape (several splits)
])
def test_block_attention_vs_oracle(B, S, Hq, Hkv, D, T, stride):
    _attn_case(B, S, Hq, Hkv, D, T, stride, seed=T + 13 * B)


@pytest.mark.parametrize("B,S,Hq,Hkv,D,T,stride", [
    (32, 16, 8, 2, 128, 1000, 1024),  # tcgen05 path: 64 pairs, two context splits of four tiles
    (3, 16, 4, 1, 64, 700, 768),      # mma.sync path
])
def test_block_attention_with_growing_keys(B, S, Hq, Hkv, D, T, stride):
    # later tiles' scores exceed the earlier maxima by far: the kernels move
    # their reference maxima and rescale what they accumulated (the tcgen05
    # kernel only within a work item, hence enough pairs for multi-tile items)
    _attn_case(B, S, Hq, Hkv, D, T, stride, seed=29, key_growth=4.0)


def test_block_attention_microbench_size_sampled():
    """The full microbenchmark shape (B=64, T=8192, 32/8 heads x 128).  Every
    (sequence, kv head) pair is checked against an fp32 torch statement of the
    same attention on the device (TF32 off), and pairs spread over the
    persistent schedule -- the first and last pairs, both neighbours of the
    middle, and those at the ends of the CTAs' item lists -- against the
    oracle, computed one pair at a time on the host."""
    from block_wise_masked_dd_b300.decoder import block_attention
    cfg = synth.ATTN_MICRO
    B, S, Hq, Hkv, D, T = cfg.batch, cfg.block, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ctx_len
    g = synth.torch_generator(11, "cuda")
    qkv = synth.torch_normal_bf16((B * S, cfg.qkv_width), 1.0, g, "cuda")
    kc = synth.torch_normal_bf16((B, Hkv, T, D), 1.0, g, "cuda")
    vc = synth.torch_normal_bf16((B, Hkv, T, D), 1.0, g, "cuda")
    out = block_attention(qkv, kc, vc, T, B, S, Hq, Hkv, D)
    torch.cuda.synchronize()
    G = Hq // Hkv
    got_all = out.float().reshape(B, S, Hkv, G, D)
    # every pair, fp32 on the device: one softmax over [context | block] keys
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        x = qkv.float().reshape(B, S, Hq + 2 * Hkv, D)
        worst = 0.0
        for b0 in range(0, B, 8):
            q = x[b0:b0 + 8, :, :Hq].reshape(-1, S, Hkv, G, D).permute(0, 2, 3, 1, 4)      # [b, kvh, g, i, d]
            kb = x[b0:b0 + 8, :, Hq:Hq + Hkv].permute(0, 2, 1, 3)                           # [b, kvh, S, d]
            vb = x[b0:b0 + 8, :, Hq + Hkv:].permute(0, 2, 1, 3)
            keys = torch.cat([kc[b0:b0 + 8].float(), kb], dim=2)                           # [b, kvh, T+S, d]
            vals = torch.cat([vc[b0:b0 + 8].float(), vb], dim=2)
            sc = torch.einsum("bhgid,bhjd->bhgij", q, keys) / np.sqrt(D)
            ref = torch.einsum("bhgij,bhjd->bhgid", torch.softmax(sc, dim=-1), vals)        # [b, kvh, g, i, d]
            got = got_all[b0:b0 + 8].permute(0, 2, 3, 1, 4)
            err = (got - ref).abs() - (TOL_ATTN + TOL_ATTN * ref.abs())
            worst = max(worst, float(err.max()))
        assert worst <= 0, f"attention outside tolerance by {worst} against the fp32 device statement"
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    pairs = [0, 1, 255, 256, 443, 444, B * Hkv - 2, B * Hkv - 1]
    for pair in pairs:
        b, kvh = divmod(pair, Hkv)
        rows = qkv[b * S:(b + 1) * S].float().cpu().numpy()
        q = rows[:, :Hq * D].reshape(S, Hq, D)[:, kvh * G:(kvh + 1) * G]
        kb = rows[:, (Hq + kvh) * D:(Hq + kvh + 1) * D].reshape(S, 1, D)
        vb = rows[:, (Hq + Hkv + kvh) * D:(Hq + Hkv + kvh + 1) * D].reshape(S, 1, D)
        want = oracle.block_attention(q, kb, vb, kc[b, kvh:kvh + 1].float().cpu().numpy(),
                                      vc[b, kvh:kvh + 1].float().cpu().numpy())
        got = bf16_to_f32(out[b * S:(b + 1) * S]).reshape(S, Hq, D)[:, kvh * G:(kvh + 1) * G]
        close(got, want, TOL_ATTN, f"attention b={b} kvh={kvh}", rel_rms=3e-3)


# ------------------------------------------------------- LM head + select

def _select_case(rows, H, V, seed, sample=None):
    from block_wise_masked_dd_b300.decoder import lmhead_select
    x = synth.make_activations(rows, H, seed=seed)
    w = synth.make_activations(V, H, seed=seed + 1, std=synth.LOGIT_STD / np.sqrt(H))
    conf, arg = lmhead_select(to_dev(x), to_dev(w))
    torch.cuda.synchronize()
    idx = np.arange(rows) if sample is None else np.asarray(sample)
    x32 = synth.bf16_bits_to_f32(x)[idx]
    w32 = synth.bf16_bits_to_f32(w)
    c_want, a_want, logits = oracle.lm_head_select(x32, w32)
    close(conf.cpu().numpy()[idx], c_want, TOL_CONF, "confidence")
    tie = oracle.near_tie_flags(logits, c_want, 2.0)  # gamma out of range: logit-gap flags only
    a = arg.cpu().numpy()[idx]
    assert ((a == a_want) | tie).all(), f"argmax differs at rows {idx[(a != a_want) & ~tie][:8]}"
    assert (a >= 0).all() and (a < V).all()


@pytest.mark.parametrize("rows,H,V", [(16, 256, 4096), (128, 2048, 32768), (200, 512, 8192), (384, 1024, 2048)])
def test_lmhead_select_vs_oracle(rows, H, V):
    _select_case(rows, H, V, seed=rows + V)


def test_lmhead_select_microbench_size_sampled():
    """1024 rows x 4096 x 131072 (the LM-head microbenchmark), 48 rows sampled
    across all eight 128-row tiles."""
    sample = list(range(0, 1024, 64)) + list(range(1, 1024, 61)) + [127, 128, 1023]
    _select_case(1024, 4096, 131072, seed=5, sample=sorted(set(sample)))


def test_lmhead_select_equal_logits():
    """All-zero weights: every logit ties, conf = 1/V and the argmax is id 0."""
    from block_wise_masked_dd_b300.decoder import lmhead_select
    x = torch.randn(32, 512, device="cuda").to(torch.bfloat16)
    w = torch.zeros(4096, 512, device="cuda", dtype=torch.bfloat16)
    conf, arg = lmhead_select(x, w)
    assert torch.allclose(conf, torch.full_like(conf, 1 / 4096), rtol=1e-5)
    assert (arg == 0).all()


# ------------------------------------------------------------------ commit

@pytest.mark.parametrize("gamma", [0.0, 0.5, 0.8, 0.95, 1.5])
@pytest.mark.parametrize("mode", [0, 1, 2 | (1 << 8), 2 | (3 << 8), 2 | (16 << 8), 3 | (1 << 8), 3 | (5 << 8),
                                  3 | (16 << 8)])
def test_commit_bit_exact(gamma, mode):
    """Every commit mode (threshold, mock-AR, top-k with k = 1, 3, 16, fixed
    steps with N = 1, 5, 16) against the oracle's rule, bit-exact."""
    from block_wise_masked_dd_b300.decoder import commit
    rng = np.random.default_rng(int(gamma * 100) + mode)
    B, S = 64, 16
    conf = rng.uniform(0, 1, (B, S)).astype(np.float32)
    conf[3] = 0.8                      # ties at exactly gamma and among themselves
    conf[4, :8] = 0.3
    arg = rng.integers(0, 32768, (B, S)).astype(np.int32)
    tok = rng.integers(0, 32768, (B, S)).astype(np.int32)
    mask = rng.integers(0, 1 << S, B).astype(np.uint32)
    mask[0] = 0
    mask[1] = 0xFFFF
    mask[2] = 1 << 15
    g = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    t_d, m_d = g(tok), g(mask.view(np.int32))
    n, rem = commit(g(conf), g(arg), t_d, m_d, gamma, mode)
    torch.cuda.synchronize()
    w_tok, w_mask, w_n, _ = oracle.commit(conf, arg, tok, mask, gamma, mode, S)
    assert (t_d.cpu().numpy() == w_tok).all()
    assert (m_d.cpu().numpy().view(np.uint32) == w_mask).all()
    assert (n.cpu().numpy() == w_n).all()
    assert rem.item() == sum(bin(int(v)).count("1") for v in w_mask)


# ---------------------------------------------------------------- timeout

def test_bounded_wait_reports_timeout():
    from block_wise_masked_dd_b300 import binding as B
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(B.DDError) as e:
        B.dd_test_wait_timeout(2000, status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert e.value.status == B.DD_ERR_DEVICE_TIMEOUT
    # the context is still usable afterwards
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum()) == 8.0


def test_single_kernel_calls_clear_their_status_word():
    """dd_block_attention, dd_lmhead_select and dd_gemm clear the status word
    in the first 4 bytes of their workspace, and no wait expires on these
    inputs, so each leaves it 0 (a stale non-zero word is planted first)."""
    from block_wise_masked_dd_b300 import binding as B
    from block_wise_masked_dd_b300.decoder import BlockAttention, LmHeadSelect, workspace_status
    dev = "cuda"
    g = torch.Generator(device=dev).manual_seed(7)
    nb, S, Hq, Hkv, D, T, stride = 2, 16, 8, 2, 128, 300, 384  # the tcgen05 context path and its merge
    op = BlockAttention(nb, S, Hq, Hkv, D, T, stride, dev)
    op.workspace[:4].fill_(0xFF)
    qkv = torch.randn(nb * S, (Hq + 2 * Hkv) * D, device=dev, generator=g).bfloat16()
    kc = torch.randn(nb, Hkv, stride, D, device=dev, generator=g).bfloat16()
    vc = torch.randn(nb, Hkv, stride, D, device=dev, generator=g).bfloat16()
    out = torch.empty(nb * S, Hq * D, dtype=torch.bfloat16, device=dev)
    op(qkv, kc, vc, out)
    assert op.status() == 0 and torch.isfinite(out.float()).all()

    rows, H, V = 128, 256, 4096
    lm = LmHeadSelect(rows, H, V, dev)
    lm.workspace[:4].fill_(0xFF)
    x = torch.randn(rows, H, device=dev, generator=g).bfloat16()
    w = torch.randn(V, H, device=dev, generator=g).bfloat16()
    conf = torch.empty(rows, dtype=torch.float32, device=dev)
    arg = torch.empty(rows, dtype=torch.int32, device=dev)
    lm(x, w, conf, arg)
    assert lm.status() == 0 and bool(((arg >= 0) & (arg < V)).all())

    n, k = 256, 256
    ws_bytes = B.dd_gemm_workspace_size(rows, n, k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    ws[:4].fill_(0xFF)
    wg = torch.randn(n, k, device=dev, generator=g).bfloat16()
    y = torch.empty(rows, n, dtype=torch.float32, device=dev)
    B.dd_gemm(rows, n, k, x.data_ptr(), wg.data_ptr(), y.data_ptr(), ws.data_ptr(), ws_bytes,
              torch.cuda.current_stream().cuda_stream)
    assert workspace_status(ws) == 0
    torch.testing.assert_close(y, x.float() @ wg.float().t(), rtol=1e-2, atol=1e-2)
