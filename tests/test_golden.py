"""The oracle against the text fixtures under tests/golden/ (no GPU):
hand-derived commit-rule cases, and the oracle's own tiny-workload decode
recorded by tests/golden/make_golden.py (a guard against unannounced changes
to the oracle's arithmetic)."""
import numpy as np
import pytest

import oracle
from tests.golden_io import commit_cases, near_tie_cases, near_tie_logits, tiny_decode_cases
from tests.golden.make_golden import decode, tiny_model


@pytest.mark.parametrize("case", list(commit_cases()), ids=lambda c: c["name"])
def test_commit_rule_cases(case):
    S = 16
    conf = case["conf"].reshape(1, S)
    arg = (100 + np.arange(S, dtype=np.int32)).reshape(1, S)
    tokens = np.full((1, S), 7, np.int32)
    mask = np.array([case["mask"]], np.uint32)
    tok, m, n, _ = oracle.commit(conf, arg, tokens, mask, case["gamma"], case["mode"], S)
    assert int(m[0]) == case["mask_after"]
    assert int(n[0]) == len(case["committed"])
    for i in range(S):
        assert tok[0, i] == (100 + i if i in case["committed"] else 7)


@pytest.mark.parametrize("case", list(near_tie_cases()), ids=lambda c: c["name"])
def test_near_tie_cases(case):
    """The oracle's near-tie flags equal the hand-derived ones."""
    S = 16
    flags = oracle.near_tie_positions(near_tie_logits(case["gap"]), case["conf"].reshape(1, S),
                                      np.array([case["mask"]], np.uint32), case["gamma"], case["mode"], S)
    assert sorted(np.nonzero(flags[0])[0].tolist()) == case["flagged"]


@pytest.fixture(scope="module")
def model():
    return tiny_model()


@pytest.mark.parametrize("case", list(tiny_decode_cases()), ids=lambda c: f"g{c['gamma']}_m{c['mode']}")
def test_oracle_reproduces_tiny_fixture(model, case):
    rec = decode(model, case["gamma"], case["mode"])
    assert rec["steps"] == case["steps"]
    assert rec["commits"] == case["commits"].tolist()
    assert rec["tokens"] == case["tokens"].tolist()
    assert rec["arg"] == case["first_arg"].tolist()
    assert rec["tie"] == case["first_tie"].tolist()
    np.testing.assert_allclose(rec["conf"], case["first_conf"], rtol=1e-6)
