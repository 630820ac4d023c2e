"""Draft tree with dynamic-depth pruning, retrieval fill and hybrid merge (oracle).

Test infrastructure: the plain CPU definition of the tree-building stages.

Sources (see the package docstring for the page titles):

* Graft article, step summary and method paragraph (first point): the draft
  is a tree of token chains; at depth d a confidence c_d is computed and
  compared with a threshold tau_d to decide whether to prune; the
  architecture paragraph places the pruning checkpoints at d0, d1 and d5.
* Graft article, step summary and method paragraph (second point):
  retrieval starts from the root token and fills the stage's template from
  the GPU-resident adjacency table M.
* Graft article, method paragraph (third point) and architecture paragraph:
  retained draft nodes and retrieved nodes form one tree
  T_s = T_draft_s U G_ret_s with |T_s| = Kmax.
* Graft abstract: "prune-then-graft" attaches retrieved tokens to the
  positions pruning opened.

Floating-point convention.  Scores and the confidence are float32 values
(the GPU's precision): a row's log-sum-exp is computed exactly in float64
and rounded once to float32, and every later score operation is a single
float32 operation in the order written below.  Integer decisions taken from
these values are compared with the GPU bit-exactly only on inputs whose
decisions all have a margin (see ``draft_margins``).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Callable, List, Optional, Sequence

import numpy as np

F32 = np.float32
EMPTY = -1  # token of an empty tree slot (a draft slot no candidate fills)


def row_lse_topk(row: np.ndarray, k: int):
    """Log-sum-exp and top-k of one drafter logit row.

    Returns (lse, tokens, logits): lse = log(sum_v exp(row[v])) rounded to
    float32, and the k tokens with the largest logits, ordered by logit
    descending and token id ascending on ties, with their float32 logits.
    """
    x = row.astype(np.float64)
    m = float(x.max())
    lse = F32(m + math.log(float(np.exp(x - m).sum())))
    order = np.lexsort((np.arange(x.shape[0]), -x))[:k]
    return lse, order.astype(np.int64), row[order].astype(np.float32)


@dataclass
class Cand:
    """A draft candidate: one child produced by one drafter call."""
    depth: int          # depth of this node (root = 0)
    idx: int            # index among the candidates of its depth: slot * k + rank
    token: int
    score: np.float32   # cumulative log-probability along its root path
    parent: Optional["Cand"]  # None for children of the root
    path: List[int] = field(default_factory=list)  # tokens root..this node


@dataclass
class DraftResult:
    stage: int                  # pruning stage s (len(checkpoints) = not pruned)
    pool: List[Cand]            # every candidate produced before drafting stopped
    conf: List[np.float32]      # c_d for every drafter call made
    calls: int                  # number of drafter calls made


RowFn = Callable[[int, int, List[int]], np.ndarray]


def draft_tree(row_fn: RowFn, root_tok: int, cfg: dict) -> DraftResult:
    """Grow the autoregressive draft tree with dynamic-depth pruning.

    ``row_fn(d, f, path)`` returns the drafter's float32 logits for the f-th
    frontier node of call d, whose tokens from the root are ``path``.

    Readings (the pages name the steps but give no formulas):

    * Tree growth, EAGLE-style top-k: call 0 expands the root into its top-k
      children; call d >= 1 expands each of the k frontier nodes into its
      top-k children (k^2 candidates) and the next frontier is the k best of
      them by (score desc, candidate index asc).  Every candidate stays in
      the pool.  A child's score is parent score + (logit - lse).
    * Checkpoint d_s is tested after call d_s (which produced depth d_s + 1).
    * c_d is the summed probability exp(score) over the new frontier, added
      in frontier order in float32: the draft's own estimate that one of the
      depth-(d+1) nodes is accepted.
    * The gate g_s = [c_{d_s} < tau_s]; the first gated checkpoint stops
      drafting and sets the stage s.  No gate firing leaves s = number of
      checkpoints (the dense tree).
    """
    k = cfg["k"]
    checkpoints = cfg["checkpoints"]
    tau = cfg["tau"]
    root = Cand(depth=0, idx=0, token=int(root_tok), score=F32(0.0), parent=None, path=[int(root_tok)])
    frontier: List[Cand] = [root]
    pool: List[Cand] = []
    conf: List[np.float32] = []
    stage = len(checkpoints)
    calls = 0
    for d in range(cfg["D"]):
        cands: List[Cand] = []
        for f, par in enumerate(frontier):
            lse, toks, vals = row_lse_topk(row_fn(d, f, par.path), k)
            for r in range(k):
                step = F32(vals[r] - lse)
                score = F32(par.score + step)
                tok = int(toks[r])
                cands.append(Cand(depth=d + 1, idx=f * k + r, token=tok, score=score,
                                  parent=None if par is root else par, path=par.path + [tok]))
        calls += 1
        pool.extend(cands)
        frontier = sorted(cands, key=lambda c: (-float(c.score), c.idx))[:k]
        c_d = F32(0.0)
        for c in frontier:
            c_d = F32(c_d + F32(math.exp(float(c.score))))
        conf.append(c_d)
        if d in checkpoints:
            s = checkpoints.index(d)
            if c_d < F32(tau[s]):
                stage = s
                break
    return DraftResult(stage=stage, pool=pool, conf=conf, calls=calls)


def retained_draft(res: DraftResult, cfg: dict) -> List[Cand]:
    """The draft nodes kept at stage s, in tree order.

    Reading: the stage keeps the root plus the K_draft_s - 1 best pool
    candidates by (score desc, depth asc, candidate index asc); a child never
    scores above its parent, so the kept set is ancestor-closed.  Tree order
    is (depth asc, score desc, candidate index asc), so a parent always
    precedes its children.  A pool smaller than K_draft_s - 1 (possible only
    without retrieval, where K_draft_s = Kmax) is kept whole.
    """
    keep = cfg["K_draft"][res.stage] - 1
    best = sorted(res.pool, key=lambda c: (-float(c.score), c.depth, c.idx))[:keep]
    return sorted(best, key=lambda c: (c.depth, -float(c.score), c.idx))


def retrieve(root_tok: int, M_succ: np.ndarray, tmpl_parent: Sequence[int],
             tmpl_rank: Sequence[int]) -> List[int]:
    """Fill the retrieval envelope from the root token by lookups in M.

    Node j's token is M_succ[parent token][rank_j], the parent token being
    the root's for top-level nodes.  Reading for slots M does not fill: an
    empty slot (successor -1) makes the node a pad, and every child of a pad
    is a pad; pads are reported as -1 here and become token 0 in the tree,
    so |T_s| = Kmax holds whatever M contains.
    """
    out: List[int] = []
    for j in range(len(tmpl_parent)):
        p = tmpl_parent[j]
        ptok = int(root_tok) if p < 0 else out[p]
        if ptok < 0:
            out.append(-1)
            continue
        out.append(int(M_succ[ptok, tmpl_rank[j]]))
    return out


@dataclass
class Tree:
    tok: List[int]
    parent: List[int]
    depth: List[int]
    pos: List[int]
    mask: List[int]      # ancestor-or-self bitmask, bit j = node j
    stage: int
    n_draft: int         # K_draft_s (root included)


def merge(root_tok: int, draft_nodes: List[Cand], ret_tok: Sequence[int],
          tmpl_parent: Sequence[int], stage: int, L: int, cfg: dict) -> Tree:
    """Merge the retained draft and the stage's retrieval prefix into one tree.

    Node 0 is the root (the last emitted token, at position L, not yet in the
    cache); nodes 1 .. K_draft_s - 1 are the retained draft in tree order;
    the remaining K_ret_s nodes are the first K_ret_s template nodes, whose
    top-level nodes hang off the root.  Duplicate paths are kept (no dedup),
    so the tree always has Kmax nodes.  position = L + depth, and the
    ancestor mask is mask[i] = mask[parent[i]] | (1 << i).

    Reading for the "w/o retrieval" ablation (Graft article, results
    paragraph), where K_draft_s = Kmax may exceed what a pruned draft holds:
    the draft slots the pool cannot fill are empty nodes, token EMPTY (-1)
    under the root at depth 1.  No target token equals -1, so an empty node
    is never accepted, and it adds no pair to M.
    """
    Kmax = cfg["Kmax"]
    n_draft = cfg["K_draft"][stage]
    n_ret = Kmax - n_draft
    tok = [int(root_tok)]
    parent = [-1]
    depth = [0]
    where = {}
    for c in draft_nodes:
        where[id(c)] = len(tok)
        tok.append(c.token)
        parent.append(0 if c.parent is None else where[id(c.parent)])
        depth.append(c.depth)
    assert len(tok) <= n_draft
    while len(tok) < n_draft:
        tok.append(EMPTY)
        parent.append(0)
        depth.append(1)
    for j in range(n_ret):
        p = tmpl_parent[j]
        pi = 0 if p < 0 else n_draft + p
        tok.append(ret_tok[j] if ret_tok[j] >= 0 else 0)
        parent.append(pi)
        depth.append(depth[pi] + 1)
    mask = []
    for i in range(Kmax):
        mask.append((1 << i) | (mask[parent[i]] if parent[i] >= 0 else 0))
    pos = [L + d for d in depth]
    return Tree(tok=tok, parent=parent, depth=depth, pos=pos, mask=mask, stage=stage, n_draft=n_draft)


def build_tree(draft_logits_b: np.ndarray, root_tok: int, M_succ: np.ndarray, L: int, cfg: dict,
               block: bool = False):
    """Stages 1-3 for one request from slot-indexed drafter logits.

    ``draft_logits_b[d][f]`` is the drafter's logit row for the f-th frontier
    node of call d (call 0 uses slot 0, the root).  Returns (tree, draft
    result, retrieved tokens of the whole envelope).

    ``block=True`` reads a block drafter's output instead (Graft abstract and
    results paragraph: grafting applied to DFlash-style block drafting):
    ``draft_logits_b[d]`` is the one distribution the drafter gives for depth
    d + 1, which every frontier node of call d expands with the same top-k,
    cumulative scores, pruning and graft.
    """
    if block:
        res = draft_tree(lambda d, f, _path: draft_logits_b[d], root_tok, cfg)
    else:
        res = draft_tree(lambda d, f, _path: draft_logits_b[d, f], root_tok, cfg)
    nodes = retained_draft(res, cfg)
    ret = retrieve(root_tok, M_succ, cfg["tmpl_parent"], cfg["tmpl_rank"])
    tree = merge(root_tok, nodes, ret, cfg["tmpl_parent"], res.stage, L, cfg)
    return tree, res, ret


def build_tree_batch(draft_logits: np.ndarray, root_tok: np.ndarray, M_succ: np.ndarray,
                     L: np.ndarray, cfg: dict, block: bool = False) -> dict:
    """build_tree over a batch; returns dense [B][Kmax] arrays like the library's outputs."""
    B = draft_logits.shape[0]
    Kmax = cfg["Kmax"]
    out = dict(tok=np.zeros((B, Kmax), np.int32), parent=np.zeros((B, Kmax), np.int32),
               depth=np.zeros((B, Kmax), np.int32), pos=np.zeros((B, Kmax), np.int32),
               mask=np.zeros((B, Kmax), np.uint64), stage=np.zeros(B, np.int32),
               ret=np.full((B, len(cfg["tmpl_parent"])), -1, np.int32))
    results = []
    for b in range(B):
        tree, res, ret = build_tree(draft_logits[b], int(root_tok[b]), M_succ, int(L[b]), cfg, block=block)
        out["tok"][b] = tree.tok
        out["parent"][b] = tree.parent
        out["depth"][b] = tree.depth
        out["pos"][b] = tree.pos
        out["mask"][b] = np.array(tree.mask, dtype=np.uint64)
        out["stage"][b] = tree.stage
        out["ret"][b] = ret
        results.append(res)
    out["draft_results"] = results
    return out


def draft_margins(row_fn: RowFn, root_tok: int, cfg: dict) -> float:
    """Smallest float64 margin of the float-decided integer choices of draft_tree.

    Recomputes the draft in float64 (exact log-sum-exp, no float32 rounding)
    following the same decisions, and returns the smallest of

    * the score gap between adjacent candidates from different logit rows
      among the first k + 1 of each depth's frontier order (which nodes form
      the frontier, and in which slot order);
    * |c_d - tau_s| / tau_s at every checkpoint tested;
    * the score gap between adjacent candidates from different rows among the
      first K_draft_s of the final pool order, and between same-depth
      neighbours of the kept set (node numbering).

    Candidates from the same row are ordered exactly on both sides (same
    float32 logits, monotone rounding), so their gaps are not counted.  A
    caller treats integer parity as required only when the margin exceeds
    the float32 error of the GPU's scores.
    """
    k = cfg["k"]
    checkpoints = cfg["checkpoints"]
    tau = cfg["tau"]
    margin = math.inf
    frontier = [(0.0, None, [int(root_tok)])]  # (score, row id, path)
    pool = []  # (score, depth, idx, row id)
    stage = len(checkpoints)
    for d in range(cfg["D"]):
        cands = []
        for f, (ps, _rid, path) in enumerate(frontier):
            row = row_fn(d, f, path).astype(np.float64)
            m = row.max()
            lse = m + math.log(float(np.exp(row - m).sum()))
            order = np.lexsort((np.arange(row.shape[0]), -row))[:k]
            for r in range(k):
                cands.append((ps + row[order[r]] - lse, (d, f), f * k + r, path + [int(order[r])]))
        order_c = sorted(cands, key=lambda c: (-c[0], c[2]))
        for a, b in zip(order_c[: k], order_c[1: k + 1]):
            if a[1] != b[1]:
                margin = min(margin, abs(a[0] - b[0]))
        pool.extend((c[0], d + 1, c[2], c[1]) for c in cands)
        frontier = [(c[0], c[1], c[3]) for c in order_c[:k]]
        c_d = sum(math.exp(c[0]) for c in frontier)
        if d in checkpoints:
            s = checkpoints.index(d)
            margin = min(margin, abs(c_d - tau[s]) / max(tau[s], 1e-30))
            if c_d < tau[s]:
                stage = s
                break
    keep = cfg["K_draft"][stage] - 1
    order_p = sorted(pool, key=lambda c: (-c[0], c[1], c[2]))
    for a, b in zip(order_p[: keep], order_p[1: keep + 1]):
        if a[3] != b[3]:
            margin = min(margin, abs(a[0] - b[0]))
    kept = order_p[:keep]
    by_depth = {}
    for c in kept:
        by_depth.setdefault(c[1], []).append(c)
    for cs in by_depth.values():
        cs.sort(key=lambda c: -c[0])
        for a, b in zip(cs, cs[1:]):
            if a[3] != b[3]:
                margin = min(margin, abs(a[0] - b[0]))
    return margin
