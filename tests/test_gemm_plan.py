"""The tensor-core GEMM's planner (host logic, no GPU): for the decode
workloads' linear layers and the unit-test shapes, every plan the library
would launch keeps its CTAs within the SMs, its shared memory within a CTA's
limit and its pairs legal, and its schedule covers every (tile, K block) unit
exactly once, with as many partial slots as the most-cut tile has pieces (the
reduces read exactly those)."""
import pytest

import synth
from block_wise_masked_dd_b300 import binding as B

SMS = 148
SMEM_LIMIT = 227 * 1024
MAX_SPLITS = 16


def _layer_shapes(cfg):
    H, F = cfg.hidden, cfg.mlp
    qkvw = (cfg.n_q_heads + 2 * cfg.n_kv_heads) * cfg.head_dim
    R = cfg.batch * cfg.block
    W = cfg.n_kv_heads * cfg.head_dim
    return [(R, qkvw, H), (R, H, cfg.n_q_heads * cfg.head_dim), (R, 2 * F, H), (R, H, F),
            (R, cfg.n_layers * 2 * W, H), (R, 3 * W, H), (R, H, W)]


SHAPES = sorted({s for c in (synth.TINY, synth.SMALL, synth.LARGE) for s in _layer_shapes(c)} | {
    (16, 768, 256), (48, 384, 192), (128, 3072, 2048), (128, 2048, 5632), (512, 1024, 1024), (272, 256, 640),
    (272, 5632, 4096), (384, 7168, 4096), (512, 4096, 14336), (272, 384, 1024), (144, 512, 512), (160, 512, 512),
    (256, 28672, 4096), (208, 28672, 4096), (112, 28672, 4096), (16, 4096, 14336), (496, 6144, 4096)})


@pytest.fixture(scope="module")
def lib():
    return B.load()


def _runs(p):
    """The (tile, K block) units of each worker: stream-K runs of sk_units,
    or the uniform split's items (tile, split) dealt round-robin."""
    workers = p["grid"] // p["cluster"]
    base = (p["m_tiles"] // p["cluster"]) * p["n_tiles"]
    kb = p["kb_total"]
    units = []
    if p["sk_units"] > 0:
        L = p["sk_units"]
        for c in range(workers):
            units.append(set(range(c * L, min((c + 1) * L, p["sk_total"]))))
    else:
        items = base * p["splits"]
        for c in range(workers):
            u = set()
            for t in range(c, items, workers):
                split, tile = divmod(t, base)
                u |= {tile * kb + b for b in range(split * p["kb_per_split"], min(kb, (split + 1) * p["kb_per_split"]))}
            units.append(u)
    return base, units


@pytest.mark.parametrize("rows,n,k", SHAPES)
@pytest.mark.parametrize("split", [1, 0])
def test_plan_is_legal_and_covers_every_unit_once(lib, rows, n, k, split):
    p = B.dd_gemm_plan_query(rows, n, k, split)
    # launch shape and resources
    assert 1 <= p["grid"] <= SMS and p["grid"] % p["cluster"] == 0
    assert p["smem_bytes"] <= SMEM_LIMIT and p["stages"] >= 2
    assert p["bk"] in (32, 64) and p["kb_total"] * p["bk"] == k
    assert p["m_tiles"] * 128 == n
    assert p["BN"] % 16 == 0 and p["BN"] <= 256
    assert p["n_tiles"] * p["BN"] >= rows > (p["n_tiles"] - 1) * p["BN"]
    # CTA pairs: one MMA of M = 256 over two weight tiles, halves of an even row count
    assert p["cluster"] in (1, 2) and p["cg"] == p["cluster"]
    if p["cluster"] == 2:
        assert p["m_tiles"] % 2 == 0 and p["BN"] % 32 == 0 and p["BN"] > 128
    # every (tile, K block) unit exactly once
    base, runs = _runs(p)
    total = base * p["kb_total"]
    seen = [0] * total
    for r in runs:
        for u in r:
            seen[u] += 1
    assert seen == [1] * total
    # partial slots: the most pieces any tile is cut into (stream-K), or the split count
    pieces = [sum(1 for r in runs if any(t * p["kb_total"] <= u < (t + 1) * p["kb_total"] for u in r))
              for t in range(base)]
    assert 1 <= p["splits"] <= MAX_SPLITS
    if p["sk_units"] > 0:
        assert p["sk_total"] == total
        assert max(pieces) == p["splits"]
    else:
        assert p["splits"] * p["kb_per_split"] >= p["kb_total"] > (p["splits"] - 1) * p["kb_per_split"]
        assert all(x == p["splits"] for x in pieces)


@pytest.mark.parametrize("rows,n,k", [(128, 2048, 5632), (512, 4096, 14336), (272, 384, 1024)])
def test_workspace_holds_every_slot(lib, rows, n, k):
    p = B.dd_gemm_plan_query(rows, n, k, 0)  # the standalone GEMM's plan (bf16 activations)
    assert B.dd_gemm_workspace_size(rows, n, k) == 256 + p["splits"] * rows * n * 4


def test_pairs_at_the_large_decode_shape_only(lib):
    L, S = synth.LARGE, synth.SMALL
    big = B.dd_gemm_plan_query(L.batch * L.block, 2 * L.mlp, L.hidden, 1)
    small = B.dd_gemm_plan_query(S.batch * S.block, 2 * S.mlp, S.hidden, 1)
    assert big["cluster"] == 2 and big["cg"] == 2 and big["sk_units"] > 0
    assert small["cluster"] == 1 and small["sk_units"] == 0


def test_bad_shapes_are_refused(lib):
    for rows, n, k in [(8, 128, 64), (16, 100, 64), (16, 128, 32)]:
        with pytest.raises(B.DDError):
            B.dd_gemm_plan_query(rows, n, k, 1)
