"""Pins for the oracle's budget split and retrieval templates (CPU only)."""
import itertools
import math

import pytest

from oracle import config


def test_budget_closed_form_small():
    # Kmax = 6, D = 3, k = 2, checkpoints d0, d1: worked by hand in tests/golden/tree_hand_v8.json
    assert config.draft_budget(6, 3, 2, [0, 1]) == [2, 4, 6]


@pytest.mark.parametrize("Kmax,D,k", [(32, 6, 4), (64, 8, 8), (16, 4, 3), (64, 8, 16), (8, 8, 1)])
def test_budget_invariants(Kmax, D, k):
    cps = [d for d in (0, 1, 5) if d < D]
    kd = config.draft_budget(Kmax, D, k, cps)
    kr = [Kmax - x for x in kd]
    # Kmax = K_draft_s + K_ret_s and the dense stage retrieves nothing
    assert kd[-1] == Kmax and kr[-1] == 0
    # a smaller stage index hands more budget to retrieval
    assert all(a >= b for a, b in zip(kr, kr[1:]))
    # the draft never keeps more than its pool (plus root) at any stage
    for s, d in enumerate(cps):
        assert 1 <= kd[s] <= 1 + k + d * k * k


def test_budget_rejects_bad():
    with pytest.raises(ValueError):
        config.draft_budget(64, 2, 2, [0])  # dense pool 2 + 4 < 63
    with pytest.raises(ValueError):
        config.draft_budget(8, 4, 2, [1, 1])


def _all_paths(D, W):
    out = []
    for m in range(1, D + 1):
        out.extend(itertools.product(range(W), repeat=m))
    return out


@pytest.mark.parametrize("D,W,n", [(3, 3, 39), (3, 3, 10), (4, 2, 30), (2, 5, 12), (5, 1, 5)])
def test_template_matches_full_enumeration(D, W, n):
    # brute force: every path, sorted by the envelope key
    allp = sorted(_all_paths(D, W), key=lambda p: (math.prod(r + 1 for r in p), len(p), p))
    parent, rank, paths = config.retrieval_template(D, W, n)
    assert paths == allp[:n]
    for j, p in enumerate(paths):
        assert rank[j] == p[-1]
        if len(p) == 1:
            assert parent[j] == -1
        else:
            # ancestor-closed, parent earlier in the list
            assert 0 <= parent[j] < j and paths[parent[j]] == p[:-1]


def test_template_prefixes_are_stage_templates():
    cfg = config.make_config(Kmax=64, D=8, k=8, V=1000, W=16)
    assert cfg["K_draft"] == [8, 16, 48, 64]
    n = len(cfg["tmpl_parent"])
    assert n == 56
    # every stage's template is a prefix and each prefix is ancestor-closed
    for kr in cfg["K_ret"]:
        assert all(p < kr for p in cfg["tmpl_parent"][:kr])
    # the envelope starts with the rank-0 chain down to depth D
    assert cfg["tmpl_paths"][:8] == [tuple([0] * m) for m in range(1, 9)]


def test_template_too_small():
    with pytest.raises(ValueError):
        config.retrieval_template(3, 1, 4)
