"""Online update of the adjacency table M (oracle, test infrastructure).

Graft article, method paragraph (fourth point) and architecture paragraph:
M is updated continuously from the verified tree's logits.  The pages leave
M's layout and the update rule open; they are fixed here as:

* M is two int32 arrays succ[V][W] and cnt[V][W]; row t lists up to W
  successor tokens of token t ranked by (count desc, token id asc); an empty
  slot is (succ -1, cnt 0) and empty slots come last.
* One update takes a multiset of (src, dst) pairs.  For each touched row a
  successor already present gains its multiplicity; a new successor enters
  with its multiplicity as count; the row then keeps its top W entries by
  (count desc, token asc) and drops the rest.  The result depends only on
  the multiset, never on the order of the pairs.

Reading for which pairs feed the update: every node i of every verified
tree contributes (tree_tok[i], argmax_i), the target's greedy successor of
that node's token in that context; an empty node (token -1, which only the
"w/o retrieval" ablation produces) contributes nothing.

Prompt-evidence policy (Graft article, method paragraph: retrieval uses the
context's own evidence, which is what carries long contexts): M is seeded
with the prompt's bigrams at prefill, and each step adds the bigrams of the
tokens it emitted, starting from the last token emitted before the step
(the tree's root); `emitted_pairs` forms them.
"""
from __future__ import annotations

from collections import Counter
from typing import Dict

import numpy as np


def update_M(succ: np.ndarray, cnt: np.ndarray, src: np.ndarray, dst: np.ndarray):
    """Apply one multiset update; returns new (succ, cnt) arrays (inputs untouched)."""
    V, W = succ.shape
    succ = succ.copy()
    cnt = cnt.copy()
    src = np.asarray(src).reshape(-1)
    dst = np.asarray(dst).reshape(-1)
    # an empty tree node (token -1, see tree.merge) contributes no pair
    keep = src != -1
    src, dst = src[keep], dst[keep]
    if np.any((src < 0) | (src >= V) | (dst < 0) | (dst >= V)):
        raise ValueError("token id out of range")
    rows: Dict[int, Counter] = {}
    for s, t in zip(src.tolist(), dst.tolist()):
        rows.setdefault(s, Counter())[t] += 1
    for s, adds in rows.items():
        entries: Dict[int, int] = {}
        for j in range(W):
            if succ[s, j] >= 0:
                entries[int(succ[s, j])] = int(cnt[s, j])
        for t, c in adds.items():
            entries[t] = entries.get(t, 0) + c
        ranked = sorted(entries.items(), key=lambda e: (-e[1], e[0]))[:W]
        succ[s, :] = -1
        cnt[s, :] = 0
        for j, (t, c) in enumerate(ranked):
            succ[s, j] = t
            cnt[s, j] = c
    return succ, cnt


def emitted_pairs(tree_tok: np.ndarray, out_tok: np.ndarray, acc_len: np.ndarray):
    """(src, dst) bigrams of each request's emitted tokens: root -> out[0] -> ... -> out[acc_len-1]."""
    src, dst = [], []
    for b in range(len(acc_len)):
        prev = int(tree_tok[b][0])
        for t in range(int(acc_len[b])):
            src.append(prev)
            dst.append(int(out_tok[b][t]))
            prev = int(out_tok[b][t])
    return np.array(src, dtype=np.int32), np.array(dst, dtype=np.int32)


def empty_M(V: int, W: int):
    """An empty table: every slot (-1, 0)."""
    return np.full((V, W), -1, np.int32), np.zeros((V, W), np.int32)
