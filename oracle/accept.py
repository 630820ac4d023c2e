"""Greedy longest-accepted-path selection and KV compaction (oracle, test infrastructure).

Graft article, architecture paragraph, and Graft abstract: retrieved nodes
are ordinary proposals and verification is lossless.  With greedy (argmax)
decoding, lossless acceptance has a plain definition: a node is accepted
exactly when every token on its root path equals the target's argmax at the
node before it; the emitted tokens are the deepest accepted path plus the
target's argmax after it (the bonus token).

Readings: argmax ties go to the lower token id; between accepted nodes of
equal depth the lower node index wins (so a draft node beats a retrieved
duplicate).  The accepted length counts the root, so it equals the KV rows
appended to the cache and the number of tokens emitted.
"""
from __future__ import annotations

from typing import List, Sequence

import numpy as np


def accept(target_logits_b: np.ndarray, tok: Sequence[int], parent: Sequence[int], depth: Sequence[int]):
    """One request: returns (argmax [Kmax], acc_len, path [acc_len], out_tok [acc_len], bonus)."""
    Kmax = len(tok)
    return accept_from_argmax([int(np.argmax(target_logits_b[i])) for i in range(Kmax)], tok, parent, depth)


def accept_from_argmax(g: Sequence[int], tok: Sequence[int], parent: Sequence[int], depth: Sequence[int]):
    """The same acceptance given the target's argmax g[i] at every node directly."""
    Kmax = len(tok)
    g = [int(x) for x in g]
    ok = [False] * Kmax
    ok[0] = True
    for i in range(1, Kmax):
        ok[i] = ok[parent[i]] and tok[i] == g[parent[i]]
    best = 0
    for i in range(1, Kmax):
        if ok[i] and depth[i] > depth[best]:
            best = i
    path: List[int] = []
    i = best
    while i >= 0:
        path.append(i)
        i = parent[i]
    path.reverse()
    out_tok = [int(tok[p]) for p in path[1:]] + [g[best]]
    return g, len(path), path, out_tok, g[best]


def accept_batch(target_logits: np.ndarray, tree: dict) -> dict:
    """accept over a batch; arrays padded with -1 past each request's length."""
    B, Kmax = tree["tok"].shape
    res = dict(argmax=np.zeros((B, Kmax), np.int32), acc_len=np.zeros(B, np.int32),
               path=np.full((B, Kmax), -1, np.int32), out_tok=np.full((B, Kmax), -1, np.int32),
               bonus=np.zeros(B, np.int32))
    for b in range(B):
        g, n, path, out_tok, bonus = accept(target_logits[b], tree["tok"][b], tree["parent"][b], tree["depth"][b])
        res["argmax"][b] = g
        res["acc_len"][b] = n
        res["path"][b, :n] = path
        res["out_tok"][b, :n] = out_tok
        res["bonus"][b] = bonus
    return res


def compact(Kc: np.ndarray, Vc: np.ndarray, Kt: np.ndarray, Vt: np.ndarray, L: np.ndarray,
            path: np.ndarray, acc_len: np.ndarray):
    """Copy the accepted path's tree KV rows to the end of each request's cache.

    For t < acc_len[b]: cache row L[b] + t takes tree row path[b][t] (root
    first), for K and V alike.  Works on one layer's arrays in place
    ([B][Lcap][...] caches, [B][Kmax][...] tree KV); returns the new lengths
    L + acc_len.  Raises when a request would pass the cache capacity.
    """
    Lcap = Kc.shape[1]
    for b in range(L.shape[0]):
        n = int(acc_len[b])
        if L[b] + n > Lcap:
            raise ValueError("cache capacity exceeded")
        for t in range(n):
            Kc[b, L[b] + t] = Kt[b, path[b, t]]
            Vc[b, L[b] + t] = Vt[b, path[b, t]]
    return L + acc_len
