"""Budget split and stage-specific retrieval templates (oracle, test infrastructure).

Graft article, method paragraph (first and second points) and architecture
paragraph: each pruning stage s splits the fixed verification budget as
Kmax = K_draft_s + K_ret_s, a smaller s hands more budget to retrieval, and
the retrieval templates G_ret_s are prepared in advance as per-stage
prefixes of one envelope.  The pages give neither the per-stage K_draft_s nor
the template shape; the readings below fill both.
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple


def draft_budget(Kmax: int, D: int, k: int, checkpoints: Sequence[int]) -> List[int]:
    """Return K_draft_s for s = 0 .. len(checkpoints).

    Entry s < len(checkpoints) is the draft budget when drafting stops at
    checkpoint d_s (the 0-based drafter call after which c_{d_s} is tested);
    the last entry is the unpruned (dense) stage and equals Kmax, so that
    stage retrieves nothing.

    Reading (the pages name the split but give no numbers): the budget kept
    for the draft grows linearly with the depth reached,
        K_draft_s = 1 + min(|pool_s|, floor((Kmax - 1) * (d_s + 1) / D)),
    where |pool_s| = k + d_s * k^2 is the number of draft candidates the
    first d_s + 1 drafter calls produce and the leading 1 is the root.  This
    gives a smaller s more retrieval budget, as the architecture paragraph
    states.
    """
    if Kmax < 1 or D < 1 or k < 1:
        raise ValueError("Kmax, D and k must be positive")
    prev = -1
    for d in checkpoints:
        if not (prev < d < D):
            raise ValueError("checkpoints must be strictly increasing drafter calls < D")
        prev = d
    full_pool = k + (D - 1) * k * k
    if full_pool < Kmax - 1:
        raise ValueError("the dense draft tree is smaller than Kmax - 1 nodes")
    out = []
    for d in checkpoints:
        pool = k + d * k * k
        out.append(1 + min(pool, ((Kmax - 1) * (d + 1)) // D))
    out.append(Kmax)
    return out


def _rank_paths_with_product_at_most(D: int, W: int, bound: int) -> List[Tuple[int, ...]]:
    """All rank paths (r_1..r_m), 1 <= m <= D, 0 <= r_i < W, with prod(r_i + 1) <= bound."""
    found: List[Tuple[int, ...]] = []

    def extend(path: Tuple[int, ...], prod: int) -> None:
        if len(path) == D:
            return
        for r in range(W):
            p = prod * (r + 1)
            if p > bound:
                break
            child = path + (r,)
            found.append(child)
            extend(child, p)

    extend((), 1)
    return found


def template_key(path: Sequence[int]) -> Tuple[int, int, Tuple[int, ...]]:
    """Order of the template envelope: (prod(r_i + 1) asc, length asc, lexicographic asc)."""
    return (math.prod(r + 1 for r in path), len(path), tuple(path))


def retrieval_template(D: int, W: int, n: int) -> Tuple[List[int], List[int], List[Tuple[int, ...]]]:
    """The first n nodes of the retrieval envelope.

    Reading (the pages only say the per-stage templates are prefixes of one
    envelope, filled from the root by lookups in M): a template node is a
    rank path (r_1..r_m) with m <= D and r_i < W; the node's token is the
    r_m-th ranked successor in M of its parent's token (the root token for
    m = 1).  Nodes are ordered by (prod(r_i + 1), m, lexicographic), a
    likelihood proxy under a rank-Zipf prior.  A parent's key is smaller
    than any child's, so every prefix of the list is ancestor-closed and
    G_ret_s is simply its first K_ret_s entries.

    Returns (parent, rank, paths): parent[j] is the index of node j's parent
    in the list (-1 when it hangs off the root) and rank[j] = r_m.
    """
    if n < 0:
        raise ValueError("n must be non-negative")
    if n == 0:
        return [], [], []
    total = sum(W ** m for m in range(1, D + 1))
    if total < n:
        raise ValueError("fewer than n rank paths exist for this D and W")
    bound = 1
    while True:
        paths = _rank_paths_with_product_at_most(D, W, bound)
        if len(paths) >= n:
            break
        bound += 1
    paths.sort(key=template_key)
    paths = paths[:n]
    index = {p: j for j, p in enumerate(paths)}
    parent = [-1 if len(p) == 1 else index[p[:-1]] for p in paths]
    rank = [p[-1] for p in paths]
    return parent, rank, paths


def make_config(Kmax: int, D: int, k: int, V: int, W: int,
                checkpoints: Sequence[int] = (0, 1, 5), tau: float | Sequence[float] = 0.3,
                no_retrieval: bool = False) -> dict:
    """Collect the method's parameters into one dict (the oracle's view of a config).

    Checkpoints beyond the draft depth are dropped, so a shallow draft
    (D <= 5) keeps only the checkpoints it can reach.

    ``no_retrieval`` is the Graft article's "w/o retrieval" ablation (results
    paragraph).  Reading: the retrieval budget is zero at every stage,
    K_ret_s = 0, so Kmax = K_draft_s + K_ret_s hands the whole budget to the
    draft, K_draft_s = Kmax; a stage whose candidate pool holds fewer than
    Kmax - 1 nodes keeps all of them and leaves the remaining slots empty
    (see ``tree.merge``).  Pruning itself is unchanged.
    """
    cps = [d for d in checkpoints if d < D]
    if isinstance(tau, (int, float)):
        taus = [float(tau)] * len(cps)
    else:
        taus = [float(t) for t in tau][: len(cps)]
    K_draft = draft_budget(Kmax, D, k, cps)
    if no_retrieval:
        K_draft = [Kmax] * len(K_draft)
    K_ret = [Kmax - kd for kd in K_draft]
    n_tmpl = max(K_ret)
    tp, tr, paths = retrieval_template(D, W, n_tmpl)
    return dict(Kmax=Kmax, D=D, k=k, V=V, W=W, checkpoints=cps, tau=taus,
                K_draft=K_draft, K_ret=K_ret, tmpl_parent=tp, tmpl_rank=tr,
                tmpl_paths=paths)
