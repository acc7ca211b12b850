"""The C-ABI library loads, exports every symbol include/dd.h declares, and
rejects bad arguments on the host (no GPU needed)."""
import ctypes
import os
import re

import pytest

import synth
from block_wise_masked_dd_b300 import binding as B
from block_wise_masked_dd_b300 import build as libbuild
from block_wise_masked_dd_b300.decoder import config_struct

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return B.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "dd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dd_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_four_core_calls():
    syms = declared_symbols()
    for s in ("dd_init_weights", "dd_set_context_kv", "dd_denoise_step", "dd_decode_block"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    syms = declared_symbols()
    assert len(syms) >= 19
    for s in syms:
        assert hasattr(lib, s), s
    assert set(syms) <= set(B._SIGS), "binding misses a declared symbol"


def test_status_strings(lib):
    assert B.dd_status_string(0) == "ok"
    assert B.dd_status_string(B.DD_ERR_DEVICE_TIMEOUT) == "device wait timed out"


def test_workspace_size_host_only(lib):
    for cfg in (synth.TINY, synth.SMALL, synth.LARGE):
        n = B.dd_workspace_size(config_struct(cfg))
        kv = 2 * cfg.n_layers * cfg.batch * cfg.n_kv_heads * max(cfg.max_ctx, 64) * cfg.head_dim * 2
        assert kv <= n < kv + 2 ** 31


@pytest.mark.parametrize("bad,code", [
    (dict(block=33), B.DD_ERR_INVALID_ARG),
    (dict(head_dim=96), B.DD_ERR_UNSUPPORTED),
    (dict(n_kv_heads=3), B.DD_ERR_INVALID_ARG),
    (dict(vocab=1000), B.DD_ERR_UNSUPPORTED),
    (dict(hidden=200), B.DD_ERR_UNSUPPORTED),
    (dict(hidden=128), B.DD_ERR_UNSUPPORTED),                          # hidden/8 = 16 threads: half a warp
    (dict(hidden=640), B.DD_ERR_UNSUPPORTED),                          # 80 threads: 2.5 warps
    (dict(batch=1, block=8), B.DD_ERR_UNSUPPORTED),
    (dict(max_ctx=-1), B.DD_ERR_INVALID_ARG),
    (dict(batch=0), B.DD_ERR_INVALID_ARG),
    (dict(n_q_heads=32, n_kv_heads=1), B.DD_ERR_UNSUPPORTED),          # 32 query rows per key head x 16 > 128
    (dict(hidden=3072), B.DD_ERR_UNSUPPORTED),                         # above 2048 only 4096
    (dict(hidden=8192), B.DD_ERR_UNSUPPORTED),
    (dict(mlp=100), B.DD_ERR_UNSUPPORTED),
    (dict(n_q_heads=1, n_kv_heads=1), B.DD_ERR_UNSUPPORTED),           # q|k|v width 192, not a multiple of 128
    (dict(n_layers=0), B.DD_ERR_INVALID_ARG),
    (dict(rms_eps=-1.0), B.DD_ERR_INVALID_ARG),
    (dict(rms_eps=float("nan")), B.DD_ERR_INVALID_ARG),
    (dict(rope_theta=-1.0), B.DD_ERR_INVALID_ARG),
    (dict(rope_theta=float("inf")), B.DD_ERR_INVALID_ARG),
])
def test_bad_configs_rejected(lib, bad, code):
    cfg = synth.TINY.replace(**bad)
    with pytest.raises(B.DDError) as e:
        B.dd_workspace_size(config_struct(cfg))
    assert e.value.status == code
    assert B.dd_last_error()


@pytest.mark.parametrize("edge", [
    dict(block=32),                                   # the widest block the mask word holds
    dict(batch=1, block=16, max_ctx=0),               # no context at all
    dict(hidden=4096),
    dict(hidden=256, mlp=128, vocab=256),             # the smallest widths
    dict(hidden=768),                                 # 96 threads per row: three warps
    dict(n_q_heads=8, n_kv_heads=1),                  # 8 query heads per key head x 16 = 128 rows
    dict(rope_theta=10000.0),
])
def test_edge_configs_accepted(lib, edge):
    assert B.dd_workspace_size(config_struct(synth.TINY.replace(**edge))) > 0


def test_null_pointers_rejected_before_cuda(lib):
    with pytest.raises(B.DDError) as e:
        B.dd_create(config_struct(synth.TINY), 0, 1 << 30)
    assert e.value.status == B.DD_ERR_INVALID_ARG
    with pytest.raises(B.DDError):
        B.dd_init_weights(0, B.dd_weights())
    with pytest.raises(B.DDError):
        B.dd_decode_block(0, 0, 0.8, 0)
    p = B.dd_attn_problem(1, 16, 4, 3, 64, 10, 10, 0, 0, 0, 0, 0, 0)
    with pytest.raises(B.DDError):
        B.dd_block_attention_workspace_size(p)
    with pytest.raises(B.DDError) as e:
        B.dd_lmhead_select_workspace_size(16, 100, 4096)
    assert e.value.status == B.DD_ERR_UNSUPPORTED
    with pytest.raises(B.DDError):
        B.dd_commit(0, 16, 0, 0, 0, 0, 0.8, 0, 0, 0)
    with pytest.raises(B.DDError):
        B.dd_test_wait_timeout(0, 0)
    with pytest.raises(B.DDError) as e:
        B.dd_set_option(0, B.DD_OPT_FUSED_REDUCE, 1)
    assert e.value.status == B.DD_ERR_INVALID_ARG
    with pytest.raises(B.DDError) as e:
        B.dd_get_option(0, B.DD_OPT_FUSED_REDUCE)
    assert e.value.status == B.DD_ERR_INVALID_ARG


def test_workspace_holds_the_fused_layer_scratch(lib):
    """Configurations of at most 128 activation rows reserve the fused linear
    layers' partial-tile scratch (one CTA per SM, two slots of [rows][128]
    fp32 each) and counters; larger ones do not."""
    small = B.dd_workspace_size(config_struct(synth.SMALL))
    big = B.dd_workspace_size(config_struct(synth.SMALL.replace(batch=16)))
    scratch = 148 * 2 * 128 * 128 * 4
    assert small > scratch
    # doubling the batch doubles the activations but drops the scratch
    assert big < 2 * small


def test_kernel_workspace_sizes(lib):
    p = B.dd_attn_problem(64, 16, 32, 8, 128, 8192, 8192, 0, 0, 0, 0, 0, 0)
    n = B.dd_block_attention_workspace_size(p)
    assert n >= 256
    assert B.dd_lmhead_select_workspace_size(1024, 4096, 131072) >= 3 * 512 * 1024 * 4
    assert B.dd_gemm_workspace_size(128, 2048, 2048) >= 128 * 2048 * 4
