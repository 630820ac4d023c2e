"""Pins for the oracle's acceptance, KV compaction and M update (CPU only)."""
import json
import os

import numpy as np
import pytest

from oracle import accept as acc
from oracle import update_m as um

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    with open(os.path.join(GOLDEN, "accept_update_hand.json")) as f:
        return json.load(f)


def _onehot_logits(argmax, V, rng):
    lg = rng.normal(0, 1, (len(argmax), V)).astype(np.float32)
    for i, g in enumerate(argmax):
        lg[i, g] = lg[i].max() + 1
    return lg


@pytest.mark.parametrize("case", [0, 1, 2])
def test_hand_worked_accept(case):
    c = _golden()["accept"][case]
    lg = _onehot_logits(c["argmax"], c["V"], np.random.default_rng(case))
    g, n, path, out_tok, bonus = acc.accept(lg, c["tok"], c["parent"], c["depth"])
    assert g == c["argmax"] and n == c["acc_len"] and path == c["path"]
    assert out_tok == c["out_tok"] and bonus == c["bonus"]


def test_argmax_ties_to_lower_id():
    lg = np.zeros((1, 9), np.float32)
    lg[0, [2, 6]] = 5.0
    g, n, path, out_tok, bonus = acc.accept(lg, [1], [-1], [0])
    assert g == [2] and n == 1 and out_tok == [2] and bonus == 2


def test_single_node_is_plain_greedy():
    rng = np.random.default_rng(1)
    lg = rng.normal(0, 1, (1, 500)).astype(np.float32)
    g, n, path, out_tok, bonus = acc.accept(lg, [42], [-1], [0])
    assert n == 1 and path == [0] and out_tok == [int(lg[0].argmax())] == [bonus]


@pytest.mark.parametrize("seed", range(8))
def test_chain_accepts_longest_matching_prefix(seed):
    rng = np.random.default_rng(seed)
    K, V = 10, 12
    tok = rng.integers(0, V, K).tolist()
    lg = rng.normal(0, 1, (K, V)).astype(np.float32)
    m = int(rng.integers(0, K))
    for i in range(m):  # plant a match for the first m edges
        lg[i, tok[i + 1]] = lg[i].max() + 1
    parent = list(range(-1, K - 1))
    g, n, path, out_tok, bonus = acc.accept(lg, tok, parent, list(range(K)))
    # brute force: count leading positions where the chain token is the argmax at its parent
    want = 1
    while want < K and int(np.argmax(lg[want - 1])) == tok[want]:
        want += 1
    assert n == want and path == list(range(want))
    assert out_tok == tok[1:want] + [int(np.argmax(lg[want - 1]))]


def test_compaction_copies_path_rows():
    rng = np.random.default_rng(2)
    B, Lcap, K, H, d = 2, 12, 5, 2, 4
    Kc, Vc = rng.normal(size=(B, Lcap, H, d)), rng.normal(size=(B, Lcap, H, d))
    Kt, Vt = rng.normal(size=(B, K, H, d)), rng.normal(size=(B, K, H, d))
    Kc0, Vc0 = Kc.copy(), Vc.copy()
    L = np.array([3, 7])
    path = np.array([[0, 2, 4, -1, -1], [0, -1, -1, -1, -1]])
    n = np.array([3, 1])
    L2 = acc.compact(Kc, Vc, Kt, Vt, L, path, n)
    assert L2.tolist() == [6, 8]
    assert np.array_equal(Kc[0, 3:6], Kt[0, [0, 2, 4]]) and np.array_equal(Vc[1, 7], Vt[1, 0])
    untouched = np.ones((B, Lcap), bool)
    untouched[0, 3:6] = untouched[1, 7] = False
    assert np.array_equal(Kc[untouched], Kc0[untouched]) and np.array_equal(Vc[untouched], Vc0[untouched])
    with pytest.raises(ValueError):
        acc.compact(Kc, Vc, Kt, Vt, np.array([10, 0]), path, n)


def test_hand_worked_update_with_eviction():
    u = _golden()["update_M"]
    succ = np.array(u["succ_before"], np.int32)
    cnt = np.array(u["cnt_before"], np.int32)
    pairs = np.array(u["pairs"])
    s2, c2 = um.update_M(succ, cnt, pairs[:, 0], pairs[:, 1])
    assert s2.tolist() == u["succ_after"] and c2.tolist() == u["cnt_after"]


def _random_M(rng, V, W, fill):
    succ = np.full((V, W), -1, np.int32)
    cnt = np.zeros((V, W), np.int32)
    for t in range(V):
        n = int(rng.integers(0, fill + 1))
        toks = rng.choice(V, n, replace=False)
        cs = rng.integers(1, 9, n)
        order = sorted(range(n), key=lambda j: (-cs[j], toks[j]))
        succ[t, :n] = toks[order]
        cnt[t, :n] = cs[order]
    return succ, cnt


@pytest.mark.parametrize("seed", range(5))
def test_update_is_order_independent(seed):
    rng = np.random.default_rng(seed)
    V, W = 30, 4
    succ, cnt = _random_M(rng, V, W, W)
    src = rng.integers(0, V, 400)
    dst = rng.integers(0, V, 400)
    a = um.update_M(succ, cnt, src, dst)
    perm = rng.permutation(400)
    b = um.update_M(succ, cnt, src[perm], dst[perm])
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("seed", range(5))
def test_batch_equals_one_at_a_time_without_eviction(seed):
    """With room for every successor no entry is evicted, so applying the
    pairs one by one (each a one-pair update, re-ranking every time) must
    give the batch result, and the total count grows by exactly n."""
    rng = np.random.default_rng(seed)
    V, W = 12, 12
    succ, cnt = _random_M(rng, V, W, 3)
    src = rng.integers(0, V, 60)
    dst = rng.integers(0, V, 60)
    bs, bc = um.update_M(succ, cnt, src, dst)
    s, c = succ, cnt
    for a, b in zip(src, dst):
        row_s, row_c = list(s[a]), list(c[a])
        if b in row_s:
            row_c[row_s.index(b)] += 1
        else:
            row_s[row_s.index(-1)] = b
            row_c[row_s.index(b)] = 1
        ent = sorted([(x, y) for x, y in zip(row_s, row_c) if x >= 0], key=lambda e: (-e[1], e[0]))
        s = s.copy()
        c = c.copy()
        s[a] = [e[0] for e in ent] + [-1] * (W - len(ent))
        c[a] = [e[1] for e in ent] + [0] * (W - len(ent))
    assert np.array_equal(bs, s) and np.array_equal(bc, c)
    assert int(bc.sum()) == int(cnt.sum()) + 60
    # rows stay ranked with empties last
    for t in range(V):
        ent = [(x, y) for x, y in zip(bs[t], bc[t])]
        real = [e for e in ent if e[0] >= 0]
        assert ent[: len(real)] == sorted(real, key=lambda e: (-e[1], e[0]))
        assert all(e == (-1, 0) for e in ent[len(real):])


def test_update_rejects_out_of_range():
    succ, cnt = um.empty_M(5, 2)
    with pytest.raises(ValueError):
        um.update_M(succ, cnt, np.array([5]), np.array([0]))


def test_emitted_pairs_hand_example():
    """Root 7 emits 3, 9 (path) and bonus 4: bigrams 7->3, 3->9, 9->4; a request that accepted only the
    root emits its bonus: 5->6."""
    from oracle import update_m as oupd
    tree_tok = np.array([[7, 3, 9, 1], [5, 2, 2, 2]], np.int32)
    out_tok = np.array([[3, 9, 4, -1], [6, -1, -1, -1]], np.int32)
    src, dst = oupd.emitted_pairs(tree_tok, out_tok, np.array([3, 1], np.int32))
    assert list(zip(src.tolist(), dst.tolist())) == [(7, 3), (3, 9), (9, 4), (5, 6)]


def test_prompt_seeding_counts_bigrams():
    """Seeding from a token stream counts each bigram: the stream 1 2 1 2 1 3 gives row 1 = {2: 2, 3: 1}
    and row 2 = {1: 2} (closed form by counting)."""
    from oracle import update_m as oupd
    succ, cnt = oupd.empty_M(4, 2)
    toks = np.array([1, 2, 1, 2, 1, 3], np.int32)
    succ, cnt = oupd.update_M(succ, cnt, toks[:-1], toks[1:])
    assert succ[1].tolist() == [2, 3] and cnt[1].tolist() == [2, 1]
    assert succ[2].tolist() == [1, -1] and cnt[2].tolist() == [2, 0]
