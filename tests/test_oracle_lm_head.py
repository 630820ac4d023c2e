"""Pins for the lm_head argmax oracle (oracle/lm_head.py) and acceptance from a given argmax."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import accept as oacc
from oracle import lm_head as olm


def test_brute_force_exact_small():
    """Exact rational dot products in plain loops agree with the oracle on tiny inputs."""
    rng = np.random.default_rng(5)
    H = rng.integers(-8, 9, size=(6, 7)) / 8.0  # exactly representable in bf16
    W = rng.integers(-8, 9, size=(13, 7)) / 4.0
    g, mx, mg = olm.lm_head_argmax(H, W)
    for n in range(H.shape[0]):
        best, best_v = None, None
        for v in range(W.shape[0]):
            s = sum(Fraction(H[n, k]) * Fraction(W[v, k]) for k in range(H.shape[1]))
            if best is None or s > best:  # strict: the first maximum wins
                best, best_v = s, v
        assert g[n] == best_v
        assert mx[n] == float(best)


def test_planted_maxima():
    """One-hot hidden states pick out one column of W; a planted large entry fixes the argmax."""
    N, d, V = 16, 32, 500
    rng = np.random.default_rng(1)
    H = np.zeros((N, d))
    H[np.arange(N), np.arange(N)] = 1.0
    W = rng.uniform(-1, 1, size=(V, d))
    t = rng.choice(V, N, replace=False)
    W[t, np.arange(N)] = 10.0
    g, mx, mg = olm.lm_head_argmax(H, W)
    assert g.tolist() == t.tolist()
    assert np.all(mx == 10.0)
    assert np.all(mg >= 10.0 - 1.0)


def test_ties_go_to_the_lower_id():
    rng = np.random.default_rng(2)
    H = rng.normal(size=(3, 8))
    W = rng.normal(size=(20, 8)) * 0.01
    W[9] = H[1] * 3
    W[4] = W[9]  # duplicate row: identical logits
    g, mx, mg = olm.lm_head_argmax(H, W)
    assert g[1] == 4
    assert mg[1] == 0.0


def test_accept_from_argmax_matches_logits_path():
    rng = np.random.default_rng(3)
    Kmax, V = 12, 50
    parent = [-1] + [int(rng.integers(0, i)) for i in range(1, Kmax)]
    depth = [0] * Kmax
    for i in range(1, Kmax):
        depth[i] = depth[parent[i]] + 1
    tok = [int(x) for x in rng.integers(0, V, Kmax)]
    logits = rng.normal(size=(Kmax, V))
    # make the chain 0 -> 1 -> ... accepted where the tree allows it
    for i in range(1, Kmax):
        logits[parent[i], tok[i]] = 100.0 + i
    a = oacc.accept(logits, tok, parent, depth)
    b = oacc.accept_from_argmax(np.argmax(logits, axis=1), tok, parent, depth)
    assert a == b
    assert a[1] >= 2


def test_single_token_vocabulary():
    H = np.ones((3, 4))
    W = np.full((1, 4), -2.0)
    g, mx, mg = olm.lm_head_argmax(H, W)
    assert g.tolist() == [0, 0, 0] and mx.tolist() == [-8.0] * 3 and np.all(np.isinf(mg))
