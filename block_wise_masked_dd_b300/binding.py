"""ctypes binding of libdd (include/dd.h): the same names, argument marshalling only.

Pointers are passed as Python ints (device or host addresses), streams as
cudaStream_t ints (0 = legacy default stream).  Every call checks the
returned dd_status and raises DDError with the library's message.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdd.so")

DD_OK = 0
DD_ERR_INVALID_ARG = 1
DD_ERR_CUDA = 2
DD_ERR_NOT_READY = 3
DD_ERR_STEP_LIMIT = 4
DD_ERR_DEVICE_TIMEOUT = 5
DD_ERR_UNSUPPORTED = 6

DD_MODE_THRESHOLD = 0
DD_MODE_MOCK_AR = 1
DD_MODE_TOPK = 2
DD_MODE_STEPS = 3


def DD_MODE_PARAM(mode: int, param: int) -> int:
    """A commit mode with its parameter (k for top-k, N for fixed steps)."""
    return mode | (param << 8)

c_int32 = ctypes.c_int32
c_void_p = ctypes.c_void_p
c_size_t = ctypes.c_size_t
c_float = ctypes.c_float


class dd_config(ctypes.Structure):
    _fields_ = [("batch", c_int32), ("block", c_int32), ("hidden", c_int32), ("n_q_heads", c_int32),
                ("n_kv_heads", c_int32), ("head_dim", c_int32), ("n_layers", c_int32), ("mlp", c_int32),
                ("vocab", c_int32), ("max_ctx", c_int32), ("rms_eps", c_float),
                ("rope_theta", c_float)]


class dd_weights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("embed", "pos", "wqkv", "wo", "wgu", "wd", "g_attn", "g_mlp",
                                        "g_final", "lm_head")]


class dd_context_tower(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in ("embed", "g", "wqkv", "wo", "g2", "wkv")]


class dd_probe(ctypes.Structure):
    _fields_ = [("attn_out", c_void_p), ("hidden", c_void_p), ("logits", c_void_p), ("conf", c_void_p),
                ("arg", c_void_p)]


class dd_attn_problem(ctypes.Structure):
    _fields_ = [("batch", c_int32), ("block", c_int32), ("n_q_heads", c_int32), ("n_kv_heads", c_int32),
                ("head_dim", c_int32), ("ctx_len", c_int32), ("ctx_stride", c_int32), ("qkv", c_void_p),
                ("k_ctx", c_void_p), ("v_ctx", c_void_p), ("out", c_void_p), ("workspace", c_void_p),
                ("workspace_bytes", c_size_t)]


class DDError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"dd status {status}: {message}")
        self.status = status


# name -> (argtypes, restype)
_SIGS = {
    "dd_workspace_size": ([ctypes.POINTER(dd_config), ctypes.POINTER(c_size_t)], c_int32),
    "dd_create": ([ctypes.POINTER(dd_config), c_void_p, c_size_t, ctypes.POINTER(c_void_p)], c_int32),
    "dd_destroy": ([c_void_p], None),
    "dd_init_weights": ([c_void_p, ctypes.POINTER(dd_weights)], c_int32),
    "dd_set_context_kv": ([c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_void_p], c_int32),
    "dd_denoise_step": ([c_void_p, c_void_p, c_void_p, c_float, c_int32, c_void_p, c_void_p], c_int32),
    "dd_decode_block": ([c_void_p, c_void_p, c_float, c_int32, c_int32, ctypes.POINTER(c_int32), c_void_p],
                        c_int32),
    "dd_device_status": ([c_void_p, c_void_p], c_int32),
    "dd_set_context_tower": ([c_void_p, ctypes.POINTER(dd_context_tower)], c_int32),
    "dd_append_block": ([c_void_p, c_void_p, c_void_p], c_int32),
    "dd_status_string": ([c_int32], ctypes.c_char_p),
    "dd_last_error": ([], ctypes.c_char_p),
    "dd_denoise_step_probe": ([c_void_p, c_void_p, c_void_p, c_float, c_int32, c_void_p,
                               ctypes.POINTER(dd_probe), c_void_p], c_int32),
    "dd_block_attention_workspace_size": ([ctypes.POINTER(dd_attn_problem), ctypes.POINTER(c_size_t)], c_int32),
    "dd_block_attention": ([ctypes.POINTER(dd_attn_problem), c_void_p], c_int32),
    "dd_lmhead_select_workspace_size": ([c_int32, c_int32, c_int32, ctypes.POINTER(c_size_t)], c_int32),
    "dd_lmhead_select": ([c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                          c_void_p], c_int32),
    "dd_gemm_workspace_size": ([c_int32, c_int32, c_int32, ctypes.POINTER(c_size_t)], c_int32),
    "dd_gemm": ([c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p], c_int32),
    "dd_gemm_plan_query": ([c_int32, c_int32, c_int32, c_int32, c_void_p, c_int32], c_int32),
    "dd_commit": ([c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_float, c_int32, c_void_p, c_void_p,
                   c_void_p], c_int32),
    "dd_test_wait_timeout": ([c_int32, c_void_p, c_void_p], c_int32),
    "dd_lmhead_select_noalloc": ([c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p],
                                 c_int32),
    "dd_step_launch_count": ([c_void_p, ctypes.POINTER(c_int32)], c_int32),
    "dd_set_option": ([c_void_p, c_int32, c_int32], c_int32),
    "dd_get_option": ([c_void_p, c_int32, ctypes.POINTER(c_int32)], c_int32),
    "dd_profile_step": ([c_void_p, c_void_p, c_void_p, c_float, c_int32, c_void_p, c_void_p, c_int32,
                         ctypes.POINTER(c_int32), c_void_p], c_int32),
}

# dd_set_option / dd_get_option
DD_OPT_FUSED_REDUCE = 1
DD_OPT_COMPACT_SEQUENCES = 10
DD_OPT_FUSED_SPLITS = {"qkv": 2, "o": 3, "gate_up": 4, "down": 5}
DD_OPT_FUSED_GRID = {"qkv": 6, "o": 7, "gate_up": 8, "down": 9}

KIND_NAMES = ["embed_norm", "gemm_qkv", "reduce_qkv", "attention_context", "attention_merge", "gemm_o", "norm_o",
              "gemm_gate_up", "swiglu", "gemm_down", "norm_down", "lm_head_select", "select_combine", "commit"]

_lib = None


def load(path: str = LIB_PATH):
    """Load libdd.so.  Fails loudly if it has not been built: there is no
    fallback implementation."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"libdd.so not found at {path}; build it with "
                               "`python -m block_wise_masked_dd_b300.build`")
        lib = ctypes.CDLL(path)
        for name, (args, res) in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def _check(status: int):
    if status != DD_OK:
        msg = load().dd_last_error()
        raise DDError(status, msg.decode() if msg else "")


def dd_status_string(status: int) -> str:
    return load().dd_status_string(status).decode()


def dd_last_error() -> str:
    return load().dd_last_error().decode()


def dd_workspace_size(cfg: dd_config) -> int:
    n = c_size_t(0)
    _check(load().dd_workspace_size(ctypes.byref(cfg), ctypes.byref(n)))
    return n.value


def dd_create(cfg: dd_config, workspace: int, workspace_bytes: int) -> int:
    out = c_void_p(0)
    _check(load().dd_create(ctypes.byref(cfg), workspace, workspace_bytes, ctypes.byref(out)))
    return out.value


def dd_destroy(ctx: int):
    load().dd_destroy(ctx)


def dd_init_weights(ctx: int, w: dd_weights):
    _check(load().dd_init_weights(ctx, ctypes.byref(w)))


def dd_set_context_kv(ctx: int, k: int, v: int, t0: int, n: int, stream: int = 0):
    _check(load().dd_set_context_kv(ctx, k, v, t0, n, stream))


def dd_set_context_tower(ctx: int, embed: int, g: int, wqkv: int, wo: int, g2: int, wkv: int):
    t = dd_context_tower(embed, g, wqkv, wo, g2, wkv)
    _check(load().dd_set_context_tower(ctx, ctypes.byref(t)))


def dd_append_block(ctx: int, tokens: int, stream: int = 0):
    _check(load().dd_append_block(ctx, tokens, stream))


def dd_denoise_step(ctx: int, tokens: int, mask: int, gamma: float, mode: int, n_committed: int | None,
                    stream: int = 0):
    _check(load().dd_denoise_step(ctx, tokens, mask, gamma, mode, n_committed or None, stream))


def dd_decode_block(ctx: int, tokens: int, gamma: float, mode: int, max_steps: int = 0, stream: int = 0) -> int:
    steps = c_int32(0)
    _check(load().dd_decode_block(ctx, tokens, gamma, mode, max_steps, ctypes.byref(steps), stream))
    return steps.value


def dd_device_status(ctx: int, stream: int = 0):
    _check(load().dd_device_status(ctx, stream))


def dd_denoise_step_probe(ctx: int, tokens: int, mask: int, gamma: float, mode: int, n_committed: int | None,
                          probe: dd_probe, stream: int = 0):
    _check(load().dd_denoise_step_probe(ctx, tokens, mask, gamma, mode, n_committed or None,
                                        ctypes.byref(probe), stream))


def dd_block_attention_workspace_size(p: dd_attn_problem) -> int:
    n = c_size_t(0)
    _check(load().dd_block_attention_workspace_size(ctypes.byref(p), ctypes.byref(n)))
    return n.value


def dd_block_attention(p: dd_attn_problem, stream: int = 0):
    _check(load().dd_block_attention(ctypes.byref(p), stream))


def dd_lmhead_select_workspace_size(rows: int, hidden: int, vocab: int) -> int:
    n = c_size_t(0)
    _check(load().dd_lmhead_select_workspace_size(rows, hidden, vocab, ctypes.byref(n)))
    return n.value


def dd_lmhead_select(rows: int, hidden: int, vocab: int, x: int, w: int, conf: int, arg: int, workspace: int,
                     workspace_bytes: int, stream: int = 0):
    _check(load().dd_lmhead_select(rows, hidden, vocab, x, w, conf, arg, workspace, workspace_bytes, stream))


def dd_lmhead_select_noalloc(rows: int, hidden: int, vocab: int, x: int, w: int, conf: int, arg: int,
                             stream: int = 0):
    """LM head + select for callers that cannot allocate: no workspace
    argument; scratch comes from an array inside the library (see dd.h)."""
    _check(load().dd_lmhead_select_noalloc(rows, hidden, vocab, x, w, conf, arg, stream))


def dd_gemm_workspace_size(rows: int, n: int, k: int) -> int:
    out = c_size_t(0)
    _check(load().dd_gemm_workspace_size(rows, n, k, ctypes.byref(out)))
    return out.value


GEMM_PLAN_FIELDS = ("grid", "cluster", "cg", "bk", "BN", "m_tiles", "n_tiles", "kb_total", "splits", "kb_per_split",
                    "sk_units", "sk_total", "stages", "smem_bytes")


def dd_gemm_plan_query(rows: int, n: int, k: int, split_act: int = 1) -> dict:
    """The tensor-core GEMM's plan for a linear layer (host only), as a dict
    keyed by GEMM_PLAN_FIELDS (the order of dd.h)."""
    out = (c_int32 * len(GEMM_PLAN_FIELDS))()
    _check(load().dd_gemm_plan_query(rows, n, k, split_act, ctypes.cast(out, c_void_p), len(GEMM_PLAN_FIELDS)))
    return dict(zip(GEMM_PLAN_FIELDS, list(out)))


def dd_gemm(rows: int, n: int, k: int, x: int, w: int, y: int, workspace: int, workspace_bytes: int,
            stream: int = 0):
    _check(load().dd_gemm(rows, n, k, x, w, y, workspace, workspace_bytes, stream))


def dd_commit(batch: int, block: int, conf: int, arg: int, tokens: int, mask: int, gamma: float, mode: int,
              n_committed: int | None, remaining: int, stream: int = 0):
    _check(load().dd_commit(batch, block, conf, arg, tokens, mask, gamma, mode, n_committed or None, remaining,
                            stream))


def dd_test_wait_timeout(timeout_us: int, status: int, stream: int = 0):
    _check(load().dd_test_wait_timeout(timeout_us, status, stream))


def dd_step_launch_count(ctx: int) -> int:
    n = c_int32(0)
    _check(load().dd_step_launch_count(ctx, ctypes.byref(n)))
    return n.value


def dd_set_option(ctx: int, option: int, value: int):
    _check(load().dd_set_option(ctx, option, value))


def dd_get_option(ctx: int, option: int) -> int:
    v = c_int32(0)
    _check(load().dd_get_option(ctx, option, ctypes.byref(v)))
    return v.value


def dd_profile_step(ctx: int, tokens: int, mask: int, gamma: float, mode: int, cap: int = 512, stream: int = 0):
    """Returns a list of (kind name, milliseconds) for every launch of one step."""
    times = (c_float * cap)()
    kinds = (c_int32 * cap)()
    n = c_int32(0)
    _check(load().dd_profile_step(ctx, tokens, mask, gamma, mode, ctypes.cast(times, c_void_p),
                                  ctypes.cast(kinds, c_void_p), cap, ctypes.byref(n), stream))
    return [(KIND_NAMES[kinds[i]], float(times[i])) for i in range(n.value)]
