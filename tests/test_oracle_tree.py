"""Pins for the oracle's draft tree, pruning, retrieval and merge (CPU only)."""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import log_softmax, logsumexp

from oracle import config, tree as tr

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_row_lse_topk_library_and_brute_force():
    rng = np.random.default_rng(0)
    row = rng.normal(0, 2, 5000).astype(np.float32)
    row[17] = row[4000] = row.max() + 1  # exact tie at the top: lower id first
    row[23] = row[99] = np.float32(3.25)
    lse, toks, vals = tr.row_lse_topk(row, 6)
    assert abs(float(lse) - logsumexp(row.astype(np.float64))) <= 1e-6 * abs(float(lse))
    # brute force: repeatedly extract the largest remaining value, lowest id on ties
    left = list(range(len(row)))
    want = []
    for _ in range(6):
        best = left[0]
        for t in left:
            if row[t] > row[best]:
                best = t
        want.append(best)
        left.remove(best)
    assert toks.tolist() == want and toks[0] == 17 and toks[1] == 4000
    assert np.array_equal(vals, row[want])


def _rows_from_probs(V, pairs):
    p = np.zeros(V)
    rest = 1.0 - sum(q for _, q in pairs)
    others = [t for t in range(V) if t not in [t for t, _ in pairs]]
    p[others] = rest / len(others)
    for t, q in pairs:
        p[t] = q
    return np.log(p).astype(np.float32)


def _load_hand():
    with open(os.path.join(GOLDEN, "tree_hand_v8.json")) as f:
        g = json.load(f)
    V, D, k = g["V"], g["D"], g["k"]
    logits = np.zeros((1, D, k, V), np.float32)
    for key, row in g["draft_rows"].items():
        d, f = map(int, key.split("/"))
        logits[0, d, f] = _rows_from_probs(V, row["pairs"])
    succ = np.full((V, g["W"]), -1, np.int32)
    for t, row in g["M"].items():
        for j, (s, _c) in enumerate(row):
            succ[int(t), j] = s
    return g, logits, succ


@pytest.mark.parametrize("case", [0, 1, 2])
def test_hand_worked_tree(case):
    g, logits, succ = _load_hand()
    c = g["cases"][case]
    cfg = config.make_config(Kmax=g["Kmax"], D=g["D"], k=g["k"], V=g["V"], W=g["W"],
                             checkpoints=g["checkpoints"], tau=c["tau"])
    assert cfg["K_draft"] == g["K_draft"]
    assert [list(p) for p in cfg["tmpl_paths"]] == g["template_paths"]
    assert cfg["tmpl_parent"] == g["template_parent"] and cfg["tmpl_rank"] == g["template_rank"]
    t, res, ret = tr.build_tree(logits[0], g["root_tok"], succ, g["L"], cfg)
    assert res.stage == c["stage"]
    assert t.tok == c["tok"] and t.parent == c["parent"] and t.depth == c["depth"]
    assert t.mask == c["mask"] and ret == c["ret"]
    assert t.pos == [g["L"] + d for d in c["depth"]]


@pytest.mark.parametrize("case", [0, 1, 2])
def test_hand_worked_tree_without_retrieval(case):
    """The 'w/o retrieval' ablation: K_ret = 0 at every stage, the draft takes the whole budget and
    slots its pool cannot fill stay empty (hand-derived trees)."""
    g, logits, succ = _load_hand()
    c = g["no_retrieval_cases"][case]
    cfg = config.make_config(Kmax=g["Kmax"], D=g["D"], k=g["k"], V=g["V"], W=g["W"],
                             checkpoints=g["checkpoints"], tau=c["tau"], no_retrieval=True)
    assert cfg["K_draft"] == g["no_retrieval_K_draft"] and cfg["tmpl_parent"] == [] and cfg["K_ret"] == [0, 0, 0]
    t, res, ret = tr.build_tree(logits[0], g["root_tok"], succ, g["L"], cfg)
    assert res.stage == c["stage"] and ret == []
    assert t.tok == c["tok"] and t.parent == c["parent"] and t.depth == c["depth"] and t.mask == c["mask"]


@pytest.mark.parametrize("seed,tau", [(0, 0.9), (1, 0.3), (2, 0.6), (3, 0.0)])  # stages 0, 2, 1, 2
def test_without_retrieval_keeps_the_best_of_the_pool(seed, tau):
    """Without retrieval a stage's draft is the top-min(Kmax - 1, |pool|) of the pool, by path scores
    recomputed from scratch (sum of full log-softmax values along each root path), and every other
    slot is an empty node under the root."""
    _, logits, _ = _random_cfg_logits(seed)
    cfg_nr = config.make_config(Kmax=40, D=5, k=3, V=64, W=4, tau=tau, no_retrieval=True)
    rows = {}

    def row_fn(d, f, path):
        rows[tuple(path)] = (d, f)
        return logits[0, d, f]

    res = tr.draft_tree(row_fn, 5, cfg_nr)
    t = tr.merge(5, tr.retained_draft(res, cfg_nr), [], [], res.stage, 0, cfg_nr)
    lsm = {key: log_softmax(logits[0, d, f].astype(np.float64)) for key, (d, f) in rows.items()}
    # every candidate the drafter produced before stopping, scored independently
    cands = []
    for key in rows:
        for tok in np.argsort(-lsm[key], kind="stable")[: cfg_nr["k"]]:
            path = list(key) + [int(tok)]
            cands.append((sum(lsm[tuple(path[:i])][path[i]] for i in range(1, len(path))), tuple(path)))
    n_kept = min(39, len(cands))
    want = {p for _, p in sorted(cands, key=lambda x: -x[0])[:n_kept]}
    # the tree's draft nodes as root paths
    paths = []
    for i in range(1, 1 + n_kept):
        path, j = [], i
        while j >= 0:
            path.append(t.tok[j])
            j = t.parent[j]
        paths.append(tuple(reversed(path)))
    assert set(paths) == want
    assert t.tok[1 + n_kept:] == [tr.EMPTY] * (39 - n_kept)
    assert t.parent[1 + n_kept:] == [0] * (39 - n_kept) and t.depth[1 + n_kept:] == [1] * (39 - n_kept)
    if res.stage == 0:
        assert n_kept == cfg_nr["k"] < 39  # a d0 prune leaves empty slots


def test_update_skips_empty_nodes():
    """An empty tree node (token -1) adds no pair to M; any other id outside [0, V) is an error."""
    from oracle import update_m as um
    s, c = um.empty_M(10, 2)
    s2, c2 = um.update_M(s, c, np.array([3, -1, 3, -1]), np.array([4, 7, 4, 9]))
    assert s2[3].tolist() == [4, -1] and c2[3].tolist() == [2, 0] and int(c2.sum()) == 2
    with pytest.raises(ValueError):
        um.update_M(s, c, np.array([3, -2]), np.array([4, 1]))


def _random_cfg_logits(seed, B=1, Kmax=24, D=5, k=3, V=64, W=4, sharp=3.0, tau=0.3):
    rng = np.random.default_rng(seed)
    cfg = config.make_config(Kmax=Kmax, D=D, k=k, V=V, W=W, tau=tau)
    logits = (rng.normal(0, 1, (B, D, k, V)) * sharp).astype(np.float32)
    return cfg, logits, rng


@pytest.mark.parametrize("seed", range(6))
def test_frontier_is_topk_of_recomputed_path_scores(seed):
    """Each frontier is the k best candidates of its depth, scoring each
    candidate from scratch as the sum of full log-softmax values along its
    root path (an independent computation of the cumulative score)."""
    cfg, logits, _ = _random_cfg_logits(seed, tau=0.0)  # never prune: every depth is grown
    rows = {}

    def row_fn(d, f, path):
        rows[tuple(path)] = (d, f)
        return logits[0, d, f]

    res = tr.draft_tree(row_fn, 5, cfg)
    assert res.stage == len(cfg["checkpoints"]) and res.calls == cfg["D"]
    lsm = {key: log_softmax(logits[0, d, f].astype(np.float64)) for key, (d, f) in rows.items()}

    def path_score(path):
        return sum(lsm[tuple(path[:i])][path[i]] for i in range(1, len(path)))

    for d in range(1, cfg["D"] + 1):
        cands = [c for c in res.pool if c.depth == d]
        assert len(cands) == (cfg["k"] if d == 1 else cfg["k"] ** 2)
        for c in cands:
            assert abs(float(c.score) - path_score(c.path)) < 1e-4
        # the next depth's parents are exactly the k best of this depth
        if d < cfg["D"]:
            parents = {tuple(c.path[:-1]) for c in res.pool if c.depth == d + 1}
            best = sorted(cands, key=lambda c: -path_score(c.path))[: cfg["k"]]
            assert parents == {tuple(c.path) for c in best}


def test_confidence_is_total_probability_when_k_is_V():
    """With k = V the frontier after call 0 is every token, so c_0 = 1."""
    V = 6
    cfg = config.make_config(Kmax=4, D=1, k=V, V=V, W=2, checkpoints=[0], tau=0.999)
    row = np.random.default_rng(3).normal(0, 1, V).astype(np.float32)
    res = tr.draft_tree(lambda d, f, p: row, 0, cfg)
    assert abs(float(res.conf[0]) - 1.0) < 1e-6 and res.stage == 1  # 1 >= 0.999: no prune
    cfg2 = config.make_config(Kmax=4, D=1, k=V, V=V, W=2, checkpoints=[0], tau=1.001)
    assert tr.draft_tree(lambda d, f, p: row, 0, cfg2).stage == 0


def test_confidence_sums_top_k_probabilities():
    V = 10
    p = np.array([0.4, 0.25, 0.1, 0.05, 0.05, 0.05, 0.04, 0.03, 0.02, 0.01])
    row = np.log(p).astype(np.float32)
    cfg = config.make_config(Kmax=3, D=1, k=2, V=V, W=2, checkpoints=[0], tau=0.3)
    res = tr.draft_tree(lambda d, f, q: row, 0, cfg)
    assert abs(float(res.conf[0]) - 0.65) < 1e-6


@pytest.mark.parametrize("seed", range(4))
def test_tau_extremes(seed):
    cfg0, logits, _ = _random_cfg_logits(seed, tau=0.0)
    r0 = tr.draft_tree(lambda d, f, p: logits[0, d, f], 1, cfg0)
    assert r0.stage == len(cfg0["checkpoints"])  # tau = 0: never pruned, dense tree
    cfg1, _, _ = _random_cfg_logits(seed, tau=1.01)
    r1 = tr.draft_tree(lambda d, f, p: logits[0, d, f], 1, cfg1)
    assert r1.stage == 0 and r1.calls == 1  # tau > 1: always pruned at d0


@pytest.mark.parametrize("seed", range(10))
def test_tree_invariants(seed):
    rng = np.random.default_rng(100 + seed)
    sharp = [0.5, 2.0, 5.0, 8.0][seed % 4]
    cfg, logits, _ = _random_cfg_logits(seed, sharp=sharp, tau=[0.3, 0.5, 0.4])
    V, W = cfg["V"], cfg["W"]
    succ = np.full((V, W), -1, np.int32)
    for t in range(V):
        n = rng.integers(0, W + 1)
        succ[t, :n] = rng.choice(V, n, replace=False)
    L = int(rng.integers(0, 50))
    t, res, ret = tr.build_tree(logits[0], 7, succ, L, cfg)
    Kmax = cfg["Kmax"]
    # |T_s| = Kmax and K_draft_s + K_ret_s = Kmax
    assert len(t.tok) == Kmax and t.n_draft == cfg["K_draft"][res.stage]
    for i in range(1, Kmax):
        assert 0 <= t.parent[i] < i
        assert t.depth[i] == t.depth[t.parent[i]] + 1
        assert t.pos[i] == L + t.depth[i]
    # the ancestor mask equals a brute-force walk up the parent chain
    for i in range(Kmax):
        bits, j = 0, i
        while j >= 0:
            bits |= 1 << j
            j = t.parent[j]
        assert t.mask[i] == bits
    # kept draft = the K_draft_s - 1 best pool candidates by score
    kept = sorted(res.pool, key=lambda c: (-float(c.score), c.depth, c.idx))[: t.n_draft - 1]
    assert sorted(c.token for c in kept) == sorted(t.tok[1:t.n_draft])
    # each draft node's token is its parent's top-k child (same parent path)
    for c in kept:
        if c.parent is not None:
            assert c.parent in kept


def test_retrieve_chain_with_W1():
    V = 20
    succ = np.full((V, 1), -1, np.int32)
    chain = [4, 9, 2, 17, 0, 11]
    for a, b in zip(chain, chain[1:]):
        succ[a, 0] = b
    parent, rank, _ = config.retrieval_template(5, 1, 5)
    assert parent == [-1, 0, 1, 2, 3] and rank == [0] * 5
    # hand-following the rank-0 successors from the root
    assert tr.retrieve(4, succ, parent, rank) == chain[1:]
    succ[2, 0] = -1  # a gap turns the node into a pad and every descendant too
    assert tr.retrieve(4, succ, parent, rank) == [9, 2, -1, -1, -1]


def test_retrieve_empty_M_all_pads():
    cfg = config.make_config(Kmax=16, D=4, k=3, V=32, W=4, tau=1.5)  # always stage 0
    succ = np.full((32, 4), -1, np.int32)
    ret = tr.retrieve(3, succ, cfg["tmpl_parent"], cfg["tmpl_rank"])
    assert ret == [-1] * len(cfg["tmpl_parent"])
    logits = np.random.default_rng(0).normal(0, 1, (4, 3, 32)).astype(np.float32)
    t, res, _ = tr.build_tree(logits, 3, succ, 0, cfg)
    assert res.stage == 0 and len(t.tok) == 16
    # pads are token 0 and the tree still has Kmax nodes
    assert t.tok[t.n_draft:] == [0] * (16 - t.n_draft)


def test_block_draft_k1_is_the_top1_chain():
    """A block drafter with k = 1: the draft is the chain of each position's top token, and the
    confidence after call d is the product of those tokens' probabilities (closed form)."""
    V, D = 6, 3
    rows = np.array([[0.0, 3.0, 1.0, 0.0, 0.0, 0.0],
                     [2.0, 0.0, 0.0, 0.0, 4.0, 0.0],
                     [0.0, 0.0, 0.0, 5.0, 0.0, 1.0]])
    cfg = config.make_config(Kmax=4, D=D, k=1, V=V, W=2, checkpoints=[0, 1], tau=0.0)
    succ = np.full((V, 2), -1, np.int32)
    t, res, _ = tr.build_tree(rows, 2, succ, 10, cfg, block=True)
    assert t.tok == [2, 1, 4, 3] and t.parent == [-1, 0, 1, 2] and t.depth == [0, 1, 2, 3]
    p = np.exp(rows - logsumexp(rows, axis=1, keepdims=True))
    want = np.cumprod([p[0, 1], p[1, 4], p[2, 3]])
    assert np.allclose([float(c) for c in res.conf], want, rtol=1e-6)


def test_block_draft_children_come_from_the_shared_row():
    """With a block drafter every frontier node of call d expands the same top-k of row d."""
    rng = np.random.default_rng(3)
    V, D, k = 40, 4, 3
    rows = rng.normal(0, 2, (D, V))
    cfg = config.make_config(Kmax=12, D=D, k=k, V=V, W=2, checkpoints=[], tau=0.3)
    res = tr.draft_tree(lambda d, f, _p: rows[d], 0, cfg)
    top = [set(np.argsort(-rows[d], kind="stable")[:k].tolist()) for d in range(D)]
    for c in res.pool:
        assert int(c.token) in top[c.depth - 1]


def test_alternatives_reduce_to_the_oracle_without_near_ties():
    """The near-tie enumerator used by the GPU parity tests returns exactly the oracle's tree when no
    decision is near a tie (each hand case, and random drafts)."""
    from tests.tree_alternatives import same_tree, valid_trees
    g, logits, succ = _load_hand()
    for c in g["cases"]:
        cfg = config.make_config(Kmax=g["Kmax"], D=g["D"], k=g["k"], V=g["V"], W=g["W"],
                                 checkpoints=g["checkpoints"], tau=c["tau"])
        alts = valid_trees(lambda d, f, _p: logits[0, d, f], g["root_tok"], succ, g["L"], cfg, eps=1e-6)
        t, _, _ = tr.build_tree(logits[0], g["root_tok"], succ, g["L"], cfg)
        assert len(alts) == 1 and same_tree(alts[0], t)
    for seed in range(3):
        cfg, lg, _ = _random_cfg_logits(seed)
        row_fn = lambda d, f, _p: lg[0, d, f]
        m = tr.draft_margins(row_fn, 5, cfg)
        alts = valid_trees(row_fn, 5, np.full((64, 4), -1, np.int32), 0, cfg, eps=m / 2)
        t, _, _ = tr.build_tree(lg[0], 5, np.full((64, 4), -1, np.int32), 0, cfg)
        assert len(alts) == 1 and same_tree(alts[0], t)


def test_alternatives_cover_a_planted_cross_row_tie():
    """Two depth-2 candidates from different drafter rows with equal probability (0.45 x 0.5): the
    enumerator yields the oracle's tree and the one with their frontier slots swapped, whose depth-3
    children then come from the other rows."""
    from tests.tree_alternatives import same_tree, valid_trees
    V, D, k = 8, 3, 2
    rows = {(0, 0): [(3, 0.45), (5, 0.45)], (1, 0): [(1, 0.5), (2, 0.2)], (1, 1): [(4, 0.5), (6, 0.2)],
            (2, 0): [(7, 0.6), (0, 0.2)], (2, 1): [(2, 0.7), (3, 0.1)]}
    logits = np.zeros((D, k, V), np.float32)
    for (d, f), pairs in rows.items():
        logits[d, f] = _rows_from_probs(V, pairs)
    cfg = config.make_config(Kmax=6, D=D, k=k, V=V, W=2, checkpoints=[0, 1], tau=0.0)
    succ = np.full((V, 2), -1, np.int32)
    row_fn = lambda d, f, _p: logits[d, f]
    assert tr.draft_margins(row_fn, 2, cfg) < 1e-6
    alts = valid_trees(row_fn, 2, succ, 0, cfg, eps=1e-4)
    t, _, _ = tr.build_tree(logits, 2, succ, 0, cfg)
    assert same_tree(alts[0], t)
    distinct = []
    for a in alts:
        if not any(same_tree(a, b) for b in distinct):
            distinct.append(a)
    assert len(distinct) >= 2
    # in every alternative the depth-3 nodes are children of the two tied depth-2 nodes
    for a in distinct:
        d2 = {i for i in range(6) if a.depth[i] == 2}
        assert all(a.parent[i] in d2 for i in range(6) if a.depth[i] == 3)
