"""Every tree the oracle could build if its near-tied decisions went the other way.

The tree build takes integer decisions from float32 scores: which candidates
form the next frontier and in which slot order, whether a checkpoint's
confidence falls below its threshold, which pool candidates the stage keeps,
and how same-depth kept nodes are numbered.  The GPU computes a row's
log-sum-exp in float32 in its own order, the oracle exactly and then rounded,
so a decision whose margin is below the tests' MARGIN may legitimately go
either way.  For such inputs parity means: the GPU's tree is one of the trees
obtained by letting any of those near-tied decisions flip, with every other
decision taken exactly as the oracle takes it.

``valid_trees`` follows ``oracle.tree.draft_tree`` / ``retained_draft`` step
for step (same float32 arithmetic through the oracle's ``row_lse_topk``),
with one addition: at each near-tied decision it asks a ``Decisions`` object
whether to take the other branch, and a depth-first search over those
answers enumerates every combination.  Adjacent candidates from the same
logit row are never swapped: both sides order them by the same float32
logits, exactly.
"""
from __future__ import annotations

import math
from typing import Callable, List

import numpy as np

from oracle import tree as tr

F32 = np.float32


class Decisions:
    """Answers near-tie questions from a fixed prefix of choices (False past it) and counts them."""

    def __init__(self, choices):
        self.choices = list(choices)
        self.asked = 0

    def flip(self) -> bool:
        v = self.choices[self.asked] if self.asked < len(self.choices) else False
        self.asked += 1
        return v


def _row(c: tr.Cand, k: int):
    return (c.depth, c.idx // k)


def _swap_near(order: list, span: int, k: int, eps: float, dec: Decisions) -> list:
    """Offers a swap of every adjacent pair among the first span + 1 entries whose scores differ by
    less than eps and that come from different logit rows."""
    out = list(order)
    for a in range(min(span, len(out) - 1)):
        x, y = out[a], out[a + 1]
        if _row(x, k) != _row(y, k) and abs(float(x.score) - float(y.score)) < eps and dec.flip():
            out[a], out[a + 1] = y, x
    return out


def _draft(row_fn, root_tok: int, cfg: dict, eps: float, dec: Decisions):
    k, checkpoints, tau = cfg["k"], cfg["checkpoints"], cfg["tau"]
    root = tr.Cand(depth=0, idx=0, token=int(root_tok), score=F32(0.0), parent=None, path=[int(root_tok)])
    frontier, pool = [root], []
    stage = len(checkpoints)
    for d in range(cfg["D"]):
        cands = []
        for f, par in enumerate(frontier):
            lse, toks, vals = tr.row_lse_topk(row_fn(d, f, par.path), k)
            for r in range(k):
                score = F32(par.score + F32(vals[r] - lse))
                tok = int(toks[r])
                cands.append(tr.Cand(depth=d + 1, idx=f * k + r, token=tok, score=score,
                                     parent=None if par is root else par, path=par.path + [tok]))
        pool.extend(cands)
        order = sorted(cands, key=lambda c: (-float(c.score), c.idx))
        frontier = _swap_near(order, k, k, eps, dec)[:k]
        c_d = F32(0.0)
        for c in frontier:
            c_d = F32(c_d + F32(math.exp(float(c.score))))
        if d in checkpoints:
            s = checkpoints.index(d)
            gated = bool(c_d < F32(tau[s]))
            if abs(float(c_d) - tau[s]) < eps * max(tau[s], 1e-30) and dec.flip():
                gated = not gated
            if gated:
                stage = s
                break
    return stage, pool


def _retained(pool, stage: int, cfg: dict, eps: float, dec: Decisions):
    k = cfg["k"]
    keep = cfg["K_draft"][stage] - 1
    best = sorted(pool, key=lambda c: (-float(c.score), c.depth, c.idx))
    best = _swap_near(best, keep, k, eps, dec)[:keep]
    nodes = sorted(best, key=lambda c: (c.depth, -float(c.score), c.idx))
    # renumbering: same-depth neighbours from different rows may trade places
    out = list(nodes)
    for a in range(len(out) - 1):
        x, y = out[a], out[a + 1]
        if x.depth == y.depth and _row(x, k) != _row(y, k) and abs(float(x.score) - float(y.score)) < eps \
                and dec.flip():
            out[a], out[a + 1] = y, x
    # a swap never puts a child before its parent: a parent's score exceeds its child's by the
    # child's -log p, far above eps, and parents sit at a lower depth
    return out


def valid_trees(row_fn: Callable, root_tok: int, M_succ: np.ndarray, L: int, cfg: dict, eps: float,
                limit: int = 512) -> List[tr.Tree]:
    """The oracle's tree first, then every tree reachable by flipping near-tied decisions."""
    ret = tr.retrieve(root_tok, M_succ, cfg["tmpl_parent"], cfg["tmpl_rank"])

    def build(dec: Decisions) -> tr.Tree:
        stage, pool = _draft(row_fn, root_tok, cfg, eps, dec)
        nodes = _retained(pool, stage, cfg, eps, dec)
        return tr.merge(root_tok, nodes, ret, cfg["tmpl_parent"], stage, L, cfg)

    out: List[tr.Tree] = []

    def dfs(prefix):
        if len(out) >= limit:
            raise RuntimeError("too many near-tied decisions to enumerate")
        dec = Decisions(prefix)
        out.append(build(dec))
        for i in range(len(prefix), dec.asked):
            dfs(list(prefix) + [False] * (i - len(prefix)) + [True])

    dfs([])
    return out


def same_tree(a: tr.Tree, b: tr.Tree) -> bool:
    return (a.stage == b.stage and a.tok == b.tok and a.parent == b.parent and a.depth == b.depth
            and a.pos == b.pos and a.mask == b.mask)
