"""Greedy next tokens straight from the target's final hidden states (oracle, test infrastructure).

Graft article, architecture paragraph: the merged tree is verified in one
target forward, and greedy verification needs only the target's argmax at
every tree node.  That argmax is the plain definition

    g[n] = argmax_v  sum_k H[n][k] W[v][k]      (ties to the lower token id)

of the lm_head product of the final hidden states H [N][d] with the output
embedding W [V][d].  The oracle evaluates the product in float64 from the
bf16 inputs (exact products, float64 sums) with a library matrix product
and takes the first maximum of each row.  A GPU evaluates the same sums in
float32 in another order, so a row whose two largest logits lie within the
rounding of that sum can legitimately pick either; `margins` gives each
row's gap so tests compare the unique rows exactly and check the others for
validity.  Pinned by tests/test_oracle_lm_head.py (exact brute force, planted
maxima, ties).
"""
from __future__ import annotations

import numpy as np


def logits(H: np.ndarray, W: np.ndarray) -> np.ndarray:
    """float64 logits [N][V] of H [N][d] and W [V][d] (any real dtype, bf16 values as float32)."""
    return np.asarray(H, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T


def argmax_rows(lg: np.ndarray):
    """(argmax [N] int32 with ties to the lower id, max [N] float64)."""
    g = np.argmax(lg, axis=1).astype(np.int32)  # numpy returns the first maximum
    return g, lg[np.arange(lg.shape[0]), g]


def margins(lg: np.ndarray) -> np.ndarray:
    """Gap between each row's largest and second-largest logit (0 for a tie; infinite with one token)."""
    if lg.shape[1] < 2:
        return np.full(lg.shape[0], np.inf)
    top2 = np.partition(lg, -2, axis=1)[:, -2:]
    return top2[:, 1] - top2[:, 0]


def lm_head_argmax(H: np.ndarray, W: np.ndarray):
    lg = logits(H, W)
    g, mx = argmax_rows(lg)
    return g, mx, margins(lg)
