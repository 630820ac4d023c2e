"""GPU parity: every stage of the CUDA path against the CPU oracle.

Integer and index outputs (tree, stage, argmax, accepted path and tokens,
compacted KV bytes, M) must match bit-exactly; attention must satisfy the
tolerance in tests/helpers.py.  Inputs come from the seeded generators in
tree_verification_gb300.synth and are copied to the host for the oracle.
"""
import math

import numpy as np
import pytest
import torch

from oracle import accept as oacc
from oracle import attention as oatt
from oracle import tree as otree
from oracle import update_m as oupd
from tests.helpers import MARGIN, assert_attention_close, gb, initial_M, lib_cfg, mask_to_u64, oracle_cfg, to_np, \
    warm_M
from tests.tree_alternatives import same_tree, valid_trees
from tree_verification_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    gb()


def _status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _M(wl, device=DEV):
    if wl.M_init == "zipf":
        s, c = synth.zipf_M(wl.V, wl.W, wl.seed + 5)
    else:
        s, c = synth.empty_M(wl.V, wl.W)
    return torch.from_numpy(s).to(device), torch.from_numpy(c).to(device)


def _row_fns(wl, dl_gpu, block=False):
    """Per request, the drafter row of (call d, frontier slot f), read from the device lazily (a block
    drafter's row of depth d serves every slot)."""
    fns = []
    for b in range(wl.B):
        rows = {}

        def row_fn(d, f, _path, b=b, rows=rows):
            key = (d, 0 if block else f)
            if key not in rows:
                rows[key] = (dl_gpu[b, d] if block else dl_gpu[b, d, f]).cpu().numpy()
            return rows[key]

        fns.append(row_fn)
    return fns


def _oracle_tree(wl, cfg_o, dl_gpu, roots, succ_np, L, block=False):
    """Oracle tree per request, its decision margin and its drafter-row function."""
    out, margins = [], []
    fns = _row_fns(wl, dl_gpu, block)
    for b in range(wl.B):
        row_fn = fns[b]
        res = otree.draft_tree(row_fn, int(roots[b]), cfg_o)
        nodes = otree.retained_draft(res, cfg_o)
        ret = otree.retrieve(int(roots[b]), succ_np, cfg_o["tmpl_parent"], cfg_o["tmpl_rank"])
        t = otree.merge(int(roots[b]), nodes, ret, cfg_o["tmpl_parent"], res.stage, int(L[b]), cfg_o)
        out.append(t)
        margins.append(otree.draft_margins(row_fn, int(roots[b]), cfg_o))
    return out, margins, fns


def _gpu_tree(gpu, b, n_draft):
    tok, par, dep, pos = (to_np(gpu[k])[b].tolist() for k in ("tok", "parent", "depth", "pos"))
    mask = [int(x) for x in mask_to_u64(gpu["mask"])[b]]
    st = int(to_np(gpu["stage"])[b])
    return otree.Tree(tok=tok, parent=par, depth=dep, pos=pos, mask=mask, stage=st, n_draft=n_draft)


def _check_trees(gpu, trees, margins, fns, roots, succ_np, L, cfg_o):
    """Every request checked: bit-exact where every decision clears MARGIN; otherwise the GPU's tree
    must be one of the trees the oracle builds when any decision within MARGIN goes the other way.
    Returns the number of requests compared exactly."""
    exact = 0
    for b, t in enumerate(trees):
        g = _gpu_tree(gpu, b, t.n_draft)
        if margins[b] > MARGIN:
            assert same_tree(g, t), f"request {b}: tree differs from the oracle's"
            exact += 1
        else:
            alts = valid_trees(fns[b], int(roots[b]), succ_np, int(L[b]), cfg_o, eps=MARGIN)
            assert any(same_tree(g, a) for a in alts), \
                f"request {b}: tree is none of the {len(alts)} trees near-tied decisions allow"
    return exact


def _compare_tree(gpu, trees):
    tok, par, dep, pos = (to_np(gpu[k]) for k in ("tok", "parent", "depth", "pos"))
    mask, stage = mask_to_u64(gpu["mask"]), to_np(gpu["stage"])
    for b, t in enumerate(trees):
        assert stage[b] == t.stage, f"request {b}: stage {stage[b]} vs {t.stage}"
        assert tok[b].tolist() == t.tok, f"request {b}: tokens differ"
        assert par[b].tolist() == t.parent and dep[b].tolist() == t.depth and pos[b].tolist() == t.pos
        assert [int(x) for x in mask[b]] == t.mask


def _build(wl, cfg, dl, roots, succ, L):
    status = _status()
    out = gb().graft_build_tree(cfg, dl, roots.to(DEV), succ, L.to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out


@pytest.mark.parametrize("name", ["tiny", "llama3_8b", "qwen3_8b_batch", "llama31_8b_long", "qwen3_235b"])
def test_build_tree_parity(name):
    wl = synth.WORKLOADS[name]
    cfg, cfg_o = lib_cfg(wl), oracle_cfg(wl)
    dl = synth.draft_logits(wl, DEV)
    roots, L = synth.root_tokens(wl), synth.prefix_lengths(wl)
    if wl.M_init == "warm":
        succ_np = _warm_M_oracle(wl)[0]
        succ = torch.from_numpy(succ_np).to(DEV)
    else:
        succ, _ = _M(wl)
        succ_np = succ.cpu().numpy()
    gpu = _build(wl, cfg, dl, roots, succ, L)
    trees, margins, _ = _oracle_tree(wl, cfg_o, dl, roots, succ_np, L)
    assert min(margins) > MARGIN
    _compare_tree(gpu, trees)


def _peaked_wl(V, B, seed):
    return synth.WORKLOADS["llama3_8b"].scaled(V=V, B=B, seed=seed)


@pytest.mark.parametrize("V,seed", [(4096, 1), (128256, 2)])
def test_build_tree_all_stages(V, seed):
    """Confident drafts reach every pruning stage, including the dense tree."""
    wl = _peaked_wl(V, 12, seed)
    boosts = [0.0, 10.0, 13.0, 14.0, 15.0, 16.0, 17.0, 18.0, 20.0, 22.0, 25.0, 30.0]
    if V == 4096:
        boosts = [b - math.log(128256 / 4096) for b in boosts]
    cfg, cfg_o = lib_cfg(wl), oracle_cfg(wl)
    dl = synth.peaked_draft_logits(wl, DEV, boosts, seed)
    roots, L = synth.root_tokens(wl), synth.prefix_lengths(wl)
    s_np, _ = synth.zipf_M(wl.V, wl.W, seed)
    succ = torch.from_numpy(s_np).to(DEV)
    gpu = _build(wl, cfg, dl, roots, succ, L)
    trees, margins, fns = _oracle_tree(wl, cfg_o, dl, roots, s_np, L)
    exact = _check_trees(gpu, trees, margins, fns, roots, s_np, L, cfg_o)
    assert exact >= wl.B - 2, f"too many near-tie requests: {margins}"
    stages = to_np(gpu["stage"])
    assert {0, 1, 2, 3} <= {int(stages[b]) for b in range(wl.B) if margins[b] > MARGIN}


@pytest.mark.parametrize("tau", [0.0, 1.5])
def test_build_tree_tau_extremes(tau):
    wl = synth.WORKLOADS["tiny"].scaled(B=3, V=2048)
    cfg, cfg_o = lib_cfg(wl, tau=tau), oracle_cfg(wl, tau=tau)
    dl = synth.draft_logits(wl, DEV)
    roots, L = synth.root_tokens(wl), synth.prefix_lengths(wl)
    s_np, _ = synth.zipf_M(wl.V, wl.W, 3)
    succ = torch.from_numpy(s_np).to(DEV)
    gpu = _build(wl, cfg, dl, roots, succ, L)
    trees, margins, fns = _oracle_tree(wl, cfg_o, dl, roots, s_np, L)
    if tau == 0.0:
        assert min(margins) > MARGIN
    _check_trees(gpu, trees, margins, fns, roots, s_np, L, cfg_o)
    assert set(to_np(gpu["stage"]).tolist()) == ({3} if tau == 0.0 else {0})


def test_build_tree_single_node_and_empty_M():
    wl = synth.WORKLOADS["tiny"].scaled(B=2, Kmax=1, V=1000)
    cfg, cfg_o = lib_cfg(wl), oracle_cfg(wl)
    dl = synth.draft_logits(wl, DEV)
    roots, L = synth.root_tokens(wl), synth.prefix_lengths(wl)
    s_np, _ = synth.empty_M(wl.V, wl.W)
    gpu = _build(wl, cfg, dl, roots, torch.from_numpy(s_np).to(DEV), L)
    trees, _, _ = _oracle_tree(wl, cfg_o, dl, roots, s_np, L)
    _compare_tree(gpu, trees)
    wl2 = synth.WORKLOADS["tiny"].scaled(B=2, V=1000)
    cfg2, cfg2_o = lib_cfg(wl2), oracle_cfg(wl2)
    dl2 = synth.draft_logits(wl2, DEV)
    gpu2 = _build(wl2, cfg2, dl2, roots, torch.from_numpy(s_np).to(DEV), L)
    trees2, _, _ = _oracle_tree(wl2, cfg2_o, dl2, roots, s_np, L)
    _compare_tree(gpu2, trees2)
    assert all(t.tok[t.n_draft:] == [0] * (wl2.Kmax - t.n_draft) for t in trees2)


@pytest.mark.parametrize("k", [8, 16])
def test_build_tree_tied_and_masked_rows(k):
    """Drafter rows full of ties and of -inf: integer-valued logits (the top-k decided by token id among
    equal logits), an all-equal row (with k = 16 more than 32 of a warp's entries tie with its threshold,
    so the split takes the per-thread insertion path), and rows masked to a dozen finite logits (-inf
    elsewhere; -inf entries are real entries that rank after every finite one, by id)."""
    wl = synth.WORKLOADS["llama3_8b"].scaled(B=4, V=32768, k=k, seed=11)
    cfg, cfg_o = lib_cfg(wl), oracle_cfg(wl)
    g = torch.Generator(device="cpu").manual_seed(11)
    dl = torch.empty(wl.B, wl.D, wl.k, wl.V)
    dl[0] = torch.round(torch.randn(wl.D, wl.k, wl.V, generator=g) * 2.0)
    dl[1] = 0.0
    dl[2] = -math.inf
    dl[3] = torch.round(torch.randn(wl.D, wl.k, wl.V, generator=g) * 4.0) * 0.25
    for d in range(wl.D):
        for f in range(wl.k):
            ids = torch.randperm(wl.V, generator=g)[:12]
            dl[2, d, f, ids] = torch.randn(12, generator=g)
    dl = dl.to(DEV)
    roots, L = synth.root_tokens(wl), synth.prefix_lengths(wl)
    s_np, _ = synth.zipf_M(wl.V, wl.W, 11)
    succ = torch.from_numpy(s_np).to(DEV)
    gpu = _build(wl, cfg, dl, roots, succ, L)
    trees, margins, fns = _oracle_tree(wl, cfg_o, dl, roots, s_np, L)
    _check_trees(gpu, trees, margins, fns, roots, s_np, L, cfg_o)
    assert int(to_np(gpu["stage"])[2]) > 0  # the masked rows are confident: drafting goes past call 0


def test_build_tree_zero_batch():
    wl = synth.WORKLOADS["tiny"].scaled(B=0, V=1000)
    cfg = lib_cfg(wl)
    e = torch.empty(0, dtype=torch.int32, device=DEV)
    out = gb().graft_build_tree(cfg, torch.empty(0, wl.D, wl.k, wl.V, device=DEV), e, _M(wl)[0], e)
    assert out["tok"].shape == (0, wl.Kmax)


@pytest.mark.parametrize("W,seed", [(1, 0), (8, 1), (16, 2), (32, 3)])
def test_retrieve_parity(W, seed):
    wl = synth.WORKLOADS["llama3_8b"].scaled(B=20, V=5000, W=W, D=8 if W > 1 else 8, Kmax=64 if W > 1 else 9)
    cfg, cfg_o = lib_cfg(wl), oracle_cfg(wl)
    rng = np.random.default_rng(seed)
    succ = np.full((wl.V, W), -1, np.int32)
    for t in range(wl.V):  # rows filled to a random depth: exercises pads and pad children
        n = int(rng.integers(0, W + 1))
        succ[t, :n] = rng.choice(wl.V, n, replace=False)
    roots = torch.from_numpy(rng.integers(0, wl.V, wl.B).astype(np.int32))
    roots[0] = 7
    succ[7, :] = -1  # a root with an empty row: every envelope node is a pad
    ret = gb().graft_retrieve(cfg, roots.to(DEV), torch.from_numpy(succ).to(DEV))
    torch.cuda.synchronize()
    got = to_np(ret)
    for b in range(wl.B):
        want = otree.retrieve(int(roots[b]), succ, cfg_o["tmpl_parent"], cfg_o["tmpl_rank"])
        assert got[b].tolist() == want
    assert (got[0] == -1).all()


def _attention_case(B, Hq, Hkv, Kmax, Ls, Lcap, seed, layer=0):
    wl = synth.WORKLOADS["llama3_8b"].scaled(B=B, Hq=Hq, Hkv=Hkv, Kmax=Kmax, seed=seed, L=(0, 0))
    Q, Kc, Vc, Kt, Vt = synth.layer_tensors(wl, layer, DEV, Lcap=Lcap)
    rng = np.random.default_rng(seed)
    masks = np.zeros((B, Kmax), np.uint64)
    for b in range(B):  # a random tree: parent uniformly among earlier nodes
        m = [1]
        for i in range(1, Kmax):
            m.append(m[int(rng.integers(0, i))] | (1 << i))
        masks[b] = np.array(m, dtype=np.uint64)
    L = torch.tensor(Ls, dtype=torch.int32)
    return Q, Kc, Vc, Kt, Vt, L, masks


@pytest.mark.parametrize("B,Hq,Hkv,Kmax,Ls,Lcap", [
    (1, 8, 2, 32, [512], 576),                 # one 128-row block, one chunk
    (3, 8, 2, 32, [0, 1, 1500], 1600),         # empty prefix, a single key, a ragged tail
    (2, 32, 8, 64, [4096, 777], 4160),         # two row blocks, several chunks
    (2, 64, 4, 64, [2000, 63], 2048),          # group 16: eight row blocks
    (4, 16, 16, 5, [300, 64, 65, 129], 320),   # no grouping, Kmax not a multiple of 8
    (1, 8, 1, 1, [999], 1024),                 # single-node tree: decode attention
    (2, 16, 2, 48, [1500, 300], 1536),         # 384 rows: an odd tile count, split keys
    (1, 64, 4, 5, [700], 768),                 # group 16, 80 rows: one partial tile
    (2, 12, 4, 64, [1000, 3000], 3072),        # group 3: the mma.sync path
    (3, 24, 4, 40, [0, 129, 700], 768),        # group 6, 240 rows: the mma.sync path
    (1, 32, 8, 64, [3000], 32768),             # cache far past the prefix: chunks follow the length
    (2, 12, 4, 64, [2500, 100], 16384),        # the same on the mma.sync path
])
def test_attention_parity(B, Hq, Hkv, Kmax, Ls, Lcap):
    Q, Kc, Vc, Kt, Vt, L, masks = _attention_case(B, Hq, Hkv, Kmax, Ls, Lcap, seed=B * 31 + Kmax)
    status = _status()
    O = gb().graft_tree_attention(Q, Kc, Vc, Kt, Vt, L.to(DEV), torch.from_numpy(masks.view(np.int64)).to(DEV),
                                  1 / math.sqrt(128), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oatt.tree_attention(to_np(Q), to_np(Kc), to_np(Vc), to_np(Kt), to_np(Vt), L.numpy(), masks,
                              1 / math.sqrt(128))
    assert_attention_close(to_np(O), ref)


@pytest.mark.parametrize("tiles", [1, 2])
@pytest.mark.parametrize("min_chunk", [128, 384, 1000000])
@pytest.mark.parametrize("B,Hq,Hkv,Kmax,Ls,Lcap", [
    (2, 32, 8, 64, [4096, 777], 4160),
    (3, 16, 2, 48, [0, 1500, 300], 1536),      # three tiles: the last CTA pair has one
])
def test_attention_parity_tilings_chunkings(tiles, min_chunk, B, Hq, Hkv, Kmax, Ls, Lcap):
    """Both tcgen05 kernels (one and two 128-row tiles per CTA, split-key partials merged by the merge
    kernel) with key chunks of one block, of three blocks, and one chunk per request."""
    tuning = dict(tiles=tiles, min_chunk=min_chunk, persist_ctas=-1)
    Q, Kc, Vc, Kt, Vt, L, masks = _attention_case(B, Hq, Hkv, Kmax, Ls, Lcap, seed=7 * B + Kmax)
    status = _status()
    O = gb().graft_tree_attention(Q, Kc, Vc, Kt, Vt, L.to(DEV), torch.from_numpy(masks.view(np.int64)).to(DEV),
                                  1 / math.sqrt(128), status=status, tuning=tuning)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oatt.tree_attention(to_np(Q), to_np(Kc), to_np(Vc), to_np(Kt), to_np(Vt), L.numpy(), masks,
                              1 / math.sqrt(128))
    assert_attention_close(to_np(O), ref)


@pytest.mark.parametrize("ctas", [1, 3, 7])
@pytest.mark.parametrize("min_chunk", [256, 1000000])
@pytest.mark.parametrize("B,Hq,Hkv,Kmax,Ls,Lcap", [
    (5, 32, 8, 64, [4096, 0, 777, 1, 2300], 4160),   # empty and one-key prefixes, ragged tails
    (3, 16, 2, 48, [1500, 300, 129], 1536),          # 384 rows: a partial second tile
    (2, 64, 4, 64, [2000, 63], 2048),                # group 16: four tile pairs per KV head
    (1, 8, 2, 64, [1000], 1024),                     # a single request: no length ranking
    (300, 8, 2, 64, [(37 * b) % 400 for b in range(300)], 400),  # more requests than the ranking table
])
def test_attention_parity_persistent(ctas, min_chunk, B, Hq, Hkv, Kmax, Ls, Lcap):
    """The persistent two-tile kernel with a few CTAs, so each runs many work items back to back
    (direct rows and split-key partials, items that skip, items of a request past its keys)."""
    tuning = dict(tiles=2, persist_ctas=ctas, min_chunk=min_chunk)
    Q, Kc, Vc, Kt, Vt, L, masks = _attention_case(B, Hq, Hkv, Kmax, Ls, Lcap, seed=11 * B + Kmax)
    status = _status()
    O = gb().graft_tree_attention(Q, Kc, Vc, Kt, Vt, L.to(DEV), torch.from_numpy(masks.view(np.int64)).to(DEV),
                                  1 / math.sqrt(128), status=status, tuning=tuning)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oatt.tree_attention(to_np(Q), to_np(Kc), to_np(Vc), to_np(Kt), to_np(Vt), L.numpy(), masks,
                              1 / math.sqrt(128))
    assert_attention_close(to_np(O), ref)


@pytest.mark.parametrize("ctas,split", [(40, 1), (1, 0), (3, 0), (152, 1)])
@pytest.mark.parametrize("B,Hq,Hkv,Kmax,Ls,Lcap", [
    (2, 32, 8, 64, [4096, 777], 4160),               # 16 items over up to 152 CTAs: pieces of 1 to 3 blocks
    (5, 32, 8, 64, [4096, 0, 777, 1, 2300], 4160),   # empty and one-key prefixes (a tree-only item)
    (3, 64, 4, 64, [2000, 63, 1500], 2048),          # group 16: four tile pairs per KV head
])
def test_attention_parity_stream_schedule(ctas, split, B, Hq, Hkv, Kmax, Ls, Lcap):
    """The persistent stream kernel (split 1, one key chunk per request): key blocks split evenly over
    the CTAs, so items are cut into pieces merged by the last one to finish, with more CTAs than items;
    and the whole-item deal (split 0) on the same shapes."""
    tuning = dict(tiles=2, persist_ctas=ctas, min_chunk=1000000, split=split)
    Q, Kc, Vc, Kt, Vt, L, masks = _attention_case(B, Hq, Hkv, Kmax, Ls, Lcap, seed=13 * B + ctas)
    ws = torch.zeros(gb().graft_tree_attention_workspace_size(B, Hq, Hkv, Kmax, Lcap, tuning), dtype=torch.uint8,
                     device=DEV)
    ref = oatt.tree_attention(to_np(Q), to_np(Kc), to_np(Vc), to_np(Kt), to_np(Vt), L.numpy(), masks,
                              1 / math.sqrt(128))
    for call in range(2):  # the second call reuses the workspace its first call left zeroed
        status = _status()
        O = gb().graft_tree_attention(Q, Kc, Vc, Kt, Vt, L.to(DEV), torch.from_numpy(masks.view(np.int64)).to(DEV),
                                      1 / math.sqrt(128), status=status, tuning=tuning, ws=ws)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: status {int(status.item())}"
        assert_attention_close(to_np(O), ref)


@pytest.mark.parametrize("pattern", ["ramp", "jump", "fall", "cliff"])
@pytest.mark.parametrize("Hq,Hkv,tuning", [
    (32, 8, dict(tiles=1, persist_ctas=-1, min_chunk=1000000)),     # one-tile kernel, one chunk per request
    (32, 8, dict(tiles=2, persist_ctas=-1, min_chunk=1000000)),     # two-tile kernel
    (32, 8, dict(tiles=2, persist_ctas=3, min_chunk=1000000)),      # persistent kernel, items back to back
    (32, 8, dict(tiles=2, persist_ctas=40, min_chunk=1000000, split=1)),  # stream schedule, cut items
    (32, 8, None),                                                  # the default plan (split-key chunks)
    (12, 4, None),                                                  # group 3: the mma.sync path
])
def test_attention_parity_shifting_scores(pattern, Hq, Hkv, tuning):
    """Scores that shift block to block by far more than a random cache gives: every query has 8 in
    dimension 0 and a cached key at position p of a request of L keys has 16 p / L there (ramp), 0 then
    16 from L / 2 on (jump), or 16 then 0 (fall), moving a block's scores by up to 16 log2 units, or 0
    then 128 (cliff: about 130 log2 units, past the float32 range of 2^x).  The running maximum is
    raised mid-chunk and O rescaled (ramp, jump, cliff), or later blocks weigh next to nothing (fall);
    the rows' softmax within a block stays spread.  A kernel that weighs a block against the running
    maximum alone must weigh the jump and cliff blocks again with their own maximum (their weights
    pass 2^16, at the cliff overflowing to infinity)."""
    B, Kmax, Ls, Lcap = 2, 64, [3000, 1100], 3072
    Q, Kc, Vc, Kt, Vt, L, masks = _attention_case(B, Hq, Hkv, Kmax, Ls, Lcap, seed=17 + Hq + len(pattern))
    Q[..., 0] = 8.0
    for b, Lb in enumerate(Ls):
        pos = torch.arange(Lb, dtype=torch.float32, device=DEV)
        if pattern == "ramp":
            k0 = 16.0 * pos / Lb
        elif pattern == "jump":
            k0 = torch.where(pos >= Lb // 2, 16.0, 0.0)
        elif pattern == "cliff":
            k0 = torch.where(pos >= Lb // 2, 128.0, 0.0)
        else:
            k0 = torch.where(pos < Lb // 2, 16.0, 0.0)
        Kc[b, :Lb, :, 0] = k0[:, None].to(torch.bfloat16)
    status = _status()
    kw = {} if tuning is None else dict(tuning=tuning)
    if tuning is not None and tuning.get("split") == 1:
        kw["ws"] = torch.zeros(gb().graft_tree_attention_workspace_size(B, Hq, Hkv, Kmax, Lcap, tuning),
                               dtype=torch.uint8, device=DEV)
    O = gb().graft_tree_attention(Q, Kc, Vc, Kt, Vt, L.to(DEV), torch.from_numpy(masks.view(np.int64)).to(DEV),
                                  1 / math.sqrt(128), status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oatt.tree_attention(to_np(Q), to_np(Kc), to_np(Vc), to_np(Kt), to_np(Vt), L.numpy(), masks,
                              1 / math.sqrt(128))
    assert_attention_close(to_np(O), ref)


def test_attention_stream_schedule_flags_an_unzeroed_workspace():
    """Arrival counters that do not start at zero are reported (GRAFT_STATUS_WORKSPACE)."""
    B, Hq, Hkv, Kmax, Ls, Lcap = 2, 32, 8, 64, [4096, 777], 4160
    tuning = dict(tiles=2, persist_ctas=40, min_chunk=1000000, split=1)
    Q, Kc, Vc, Kt, Vt, L, masks = _attention_case(B, Hq, Hkv, Kmax, Ls, Lcap, seed=5)
    ws = torch.full((gb().graft_tree_attention_workspace_size(B, Hq, Hkv, Kmax, Lcap, tuning),), 0x7f,
                    dtype=torch.uint8, device=DEV)
    status = _status()
    gb().graft_tree_attention(Q, Kc, Vc, Kt, Vt, L.to(DEV), torch.from_numpy(masks.view(np.int64)).to(DEV),
                              1 / math.sqrt(128), status=status, tuning=tuning, ws=ws)
    torch.cuda.synchronize()
    assert int(status.item()) & gb().STATUS_WORKSPACE


def test_attention_persistent_length_past_capacity_is_flagged():
    Q, Kc, Vc, Kt, Vt, L, masks = _attention_case(2, 32, 8, 64, [700, 100], 640, seed=3)
    status = _status()
    gb().graft_tree_attention(Q, Kc, Vc, Kt, Vt, L.to(DEV), torch.from_numpy(masks.view(np.int64)).to(DEV), 0.1,
                              status=status, tuning=dict(tiles=2, persist_ctas=2))
    torch.cuda.synchronize()
    assert int(status.item()) & gb().STATUS_LENGTH


def test_attention_length_past_capacity_is_flagged():
    Q, Kc, Vc, Kt, Vt, L, masks = _attention_case(1, 8, 2, 32, [700], 640, seed=3)
    status = _status()
    gb().graft_tree_attention(Q, Kc, Vc, Kt, Vt, L.to(DEV), torch.from_numpy(masks.view(np.int64)).to(DEV), 0.1,
                              status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & gb().STATUS_LENGTH


@pytest.mark.parametrize("name,layers,reqs", [("tiny", [0], None), ("llama3_8b", [0, 31], None),
                                              ("qwen3_8b_batch", [0], "sample"),
                                              ("llama31_8b_long", [0], None), ("qwen3_235b", [0], "sample")])
def test_attention_full_size_sampled(name, layers, reqs):
    """Full-size layer calls; the oracle recomputes sampled requests: the longest, the median and the three
    shortest (the longest-first order runs those last, and the stream schedule's last CTAs hold them)."""
    wl = synth.WORKLOADS[name]
    Lcap = wl.lcap()
    L = synth.prefix_lengths(wl)
    rng = np.random.default_rng(wl.seed)
    masks = np.zeros((wl.B, wl.Kmax), np.uint64)
    for b in range(wl.B):
        m = [1]
        for i in range(1, wl.Kmax):
            m.append(m[int(rng.integers(0, i))] | (1 << i))
        masks[b] = np.array(m, dtype=np.uint64)
    mask_d = torch.from_numpy(masks.view(np.int64)).to(DEV)
    for layer in layers:
        Q, Kc, Vc, Kt, Vt = synth.layer_tensors(wl, layer, DEV, Lcap=Lcap)
        O = gb().graft_tree_attention(Q, Kc, Vc, Kt, Vt, L.to(DEV), mask_d, 1 / math.sqrt(128))
        torch.cuda.synchronize()
        if reqs == "sample":
            order = np.lexsort((np.arange(wl.B), -L.numpy()))
            reqs = sorted({int(order[0]), int(order[wl.B // 2])} | {int(x) for x in order[-3:]})
        for b in (range(wl.B) if reqs is None else reqs):
            lb = int(L[b])
            ref = oatt.tree_attention_one(to_np(Q[b]), to_np(Kc[b, :lb]), to_np(Vc[b, :lb]), to_np(Kt[b]),
                                          to_np(Vt[b]), lb, masks[b], 1 / math.sqrt(128))
            assert_attention_close(to_np(O[b]), ref)
        del Q, Kc, Vc, Kt, Vt, O
        torch.cuda.empty_cache()


def _tree_from_oracle(wl, dl, roots, succ_np, L):
    cfg_o = oracle_cfg(wl)
    trees, _, _ = _oracle_tree(wl, cfg_o, dl, roots, succ_np, L)
    tok = np.array([t.tok for t in trees], np.int32)
    par = np.array([t.parent for t in trees], np.int32)
    dep = np.array([t.depth for t in trees], np.int32)
    return tok, par, dep


@pytest.mark.parametrize("name", ["tiny", "llama3_8b", "qwen3_8b_batch", "llama31_8b_long", "qwen3_235b"])
def test_accept_compact_parity(name):
    """Acceptance and compaction on every workload; the long-context one writes past row 65536 of its
    cache (64-bit destination offsets)."""
    wl = synth.WORKLOADS[name]
    n_layers = 2
    Lcap = wl.lcap()
    dl = synth.draft_logits(wl, DEV)
    roots, L = synth.root_tokens(wl), synth.prefix_lengths(wl)
    succ_np, _ = initial_M(wl)
    tok, par, dep = _tree_from_oracle(wl, dl, roots, succ_np, L)
    tl = synth.target_logits(wl, DEV)
    synth.plant_paths(tl, tok, par, dep, synth.planted_lengths(wl))
    layers = [synth.layer_tensors(wl.scaled(L=(8, 8)), l, DEV, Lcap=Lcap) for l in range(n_layers)]
    Kc = [x[1] for x in layers]
    Vc = [x[2] for x in layers]
    Kt = [x[3] for x in layers]
    Vt = [x[4] for x in layers]
    Kc0 = [to_np(x).copy() for x in Kc]
    Vc0 = [to_np(x).copy() for x in Vc]
    ptr = lambda ts: gb().layer_pointers(ts, DEV)
    Ld = L.to(DEV)
    status = _status()
    out = gb().graft_accept_compact(tl, torch.from_numpy(tok).to(DEV), torch.from_numpy(par).to(DEV),
                                    torch.from_numpy(dep).to(DEV), ptr(Kc), ptr(Vc), ptr(Kt), ptr(Vt), n_layers,
                                    wl.Hkv, Lcap, Ld, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oacc.accept_batch(to_np(tl), dict(tok=tok, parent=par, depth=dep))
    for k in ("argmax", "acc_len", "path", "out_tok", "bonus"):
        assert np.array_equal(to_np(out[k]), ref[k]), k
    want_L = L.numpy() + ref["acc_len"]
    assert np.array_equal(to_np(Ld), want_L)
    for l in range(n_layers):
        Kc_ref, Vc_ref = Kc0[l], Vc0[l]
        oacc.compact(Kc_ref, Vc_ref, to_np(Kt[l]), to_np(Vt[l]), L.numpy().astype(np.int64), ref["path"],
                     ref["acc_len"])
        assert np.array_equal(to_np(Kc[l]), Kc_ref) and np.array_equal(to_np(Vc[l]), Vc_ref)
    if name == "qwen3_8b_batch":
        assert len(set(ref["acc_len"].tolist())) > 2  # the planted lengths really vary


def test_accept_overflow_flagged_and_skipped():
    wl = synth.WORKLOADS["tiny"].scaled(V=500)
    Lcap = 516
    dl = synth.draft_logits(wl, DEV)
    roots = synth.root_tokens(wl)
    L = torch.tensor([514], dtype=torch.int32)
    s_np, _ = synth.zipf_M(wl.V, wl.W, 1)
    tok, par, dep = _tree_from_oracle(wl, dl, roots, s_np, L)
    tl = synth.target_logits(wl, DEV)
    synth.plant_paths(tl, tok, par, dep, [5])
    Q, Kc, Vc, Kt, Vt = synth.layer_tensors(wl, 0, DEV, Lcap=Lcap)
    before = to_np(Kc).copy()
    ptr = lambda ts: gb().layer_pointers(ts, DEV)
    Ld = L.to(DEV)
    status = _status()
    out = gb().graft_accept_compact(tl, torch.from_numpy(tok).to(DEV), torch.from_numpy(par).to(DEV),
                                    torch.from_numpy(dep).to(DEV), ptr([Kc]), ptr([Vc]), ptr([Kt]), ptr([Vt]), 1,
                                    wl.Hkv, Lcap, Ld, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & gb().STATUS_CACHE_OVERFLOW
    assert int(out["acc_len"][0]) == 5 and int(Ld[0]) == 514
    assert np.array_equal(to_np(Kc), before)


def _update_case(V, W, n, seed, fill):
    rng = np.random.default_rng(seed)
    succ = np.full((V, W), -1, np.int32)
    cnt = np.zeros((V, W), np.int32)
    for t in range(V):
        k = int(rng.integers(0, fill + 1))
        toks = rng.choice(V, k, replace=False)
        cs = rng.integers(1, 6, k)
        order = sorted(range(k), key=lambda j: (-cs[j], toks[j]))
        succ[t, :k] = toks[order]
        cnt[t, :k] = cs[order]
    src = rng.integers(0, V, n).astype(np.int32)
    dst = rng.integers(0, max(2, V // 4), n).astype(np.int32)  # few successors per row: ties, duplicates
    return succ, cnt, src, dst


@pytest.mark.parametrize("V,W,n,fill,seed", [(50, 4, 400, 4, 0), (300, 16, 4096, 16, 1), (1000, 32, 1024, 10, 2),
                                             (20, 1, 200, 1, 3), (151936, 16, 4096, 0, 4)])
def test_update_M_parity(V, W, n, fill, seed):
    succ, cnt, src, dst = _update_case(V, W, n, seed, fill)
    want_s, want_c = oupd.update_M(succ, cnt, src, dst)
    for perm_seed in (None, 7):  # the device result must not depend on pair order
        s_d, c_d = torch.from_numpy(succ).to(DEV), torch.from_numpy(cnt).to(DEV)
        order = np.arange(n) if perm_seed is None else np.random.default_rng(perm_seed).permutation(n)
        status = _status()
        gb().graft_update_M(s_d, c_d, torch.from_numpy(src[order]).to(DEV), torch.from_numpy(dst[order]).to(DEV),
                            status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert np.array_equal(to_np(s_d), want_s) and np.array_equal(to_np(c_d), want_c)


@pytest.mark.parametrize("W,hot_pairs,hot_span", [(16, 6000, 2000), (32, 3000, 40000), (1, 2500, 300)])
def test_update_M_hot_row_parity(W, hot_pairs, hot_span):
    """One source token in thousands of pairs (as a token repeated over most of a batch's tree nodes): its
    row has far more new successors than a list walk should take one by one, with repeated successors
    (multiplicities, ties on count), on top of scattered background pairs."""
    V, n_bg = 151936, 2000
    rng = np.random.default_rng(W + hot_pairs)
    succ, cnt, _, _ = _update_case(V, W, 0, W, fill=min(W, 4))
    hot = 4242
    src = np.concatenate([np.full(hot_pairs, hot, np.int32), rng.integers(0, V, n_bg).astype(np.int32)])
    dst = np.concatenate([rng.integers(0, hot_span, hot_pairs), rng.integers(0, V, n_bg)]).astype(np.int32)
    want_s, want_c = oupd.update_M(succ, cnt, src, dst)
    for perm_seed in (None, 11):
        s_d, c_d = torch.from_numpy(succ).to(DEV), torch.from_numpy(cnt).to(DEV)
        order = np.arange(len(src)) if perm_seed is None else np.random.default_rng(perm_seed).permutation(len(src))
        status = _status()
        gb().graft_update_M(s_d, c_d, torch.from_numpy(src[order]).to(DEV), torch.from_numpy(dst[order]).to(DEV),
                            status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert np.array_equal(to_np(s_d), want_s) and np.array_equal(to_np(c_d), want_c)


def test_update_M_out_of_range_pairs_are_skipped():
    succ, cnt, src, dst = _update_case(40, 4, 100, 5, 2)
    src[3] = 40
    dst[9] = -2
    keep = np.ones(100, bool)
    keep[[3, 9]] = False
    want_s, want_c = oupd.update_M(succ, cnt, src[keep], dst[keep])
    s_d, c_d = torch.from_numpy(succ).to(DEV), torch.from_numpy(cnt).to(DEV)
    status = _status()
    gb().graft_update_M(s_d, c_d, torch.from_numpy(src).to(DEV), torch.from_numpy(dst).to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & gb().STATUS_TOKEN_RANGE
    assert np.array_equal(to_np(s_d), want_s) and np.array_equal(to_np(c_d), want_c)


def _warm_pairs(wl):
    """Every adjacent pair of the seeded long-context token stream."""
    stream = synth.token_stream(wl.Lmax, wl.V, wl.seed + 41)
    return synth.stream_pairs(stream)


def _warm_M_oracle(wl):
    """The oracle's table after five warm-up rounds (input for the tree parity)."""
    return warm_M(wl)


def test_update_M_long_context_warmup():
    """Five rounds of 65535 pairs each on the device equal the oracle's table."""
    wl = synth.WORKLOADS["llama31_8b_long"]
    src, dst = _warm_pairs(wl)
    s_np, c_np = synth.empty_M(wl.V, wl.W)
    s_d, c_d = torch.from_numpy(s_np).to(DEV), torch.from_numpy(c_np).to(DEV)
    sd, dd = torch.from_numpy(src).to(DEV), torch.from_numpy(dst).to(DEV)
    for _ in range(5):
        gb().graft_update_M(s_d, c_d, sd, dd)
    torch.cuda.synchronize()
    s, c = _warm_M_oracle(wl)
    assert np.array_equal(to_np(s_d), s) and np.array_equal(to_np(c_d), c)
    assert int(c.sum()) == 5 * (wl.Lmax - 1)


@pytest.mark.parametrize("V,seed", [(4096, 4), (128256, 5)])
def test_build_tree_block_draft_parity(V, seed):
    """graft_build_tree_block (one drafter row per depth, shared by the frontier) against the oracle."""
    wl = _peaked_wl(V, 12, seed)
    boosts = [0.0, 10.0, 13.0, 14.0, 15.0, 16.0, 17.0, 18.0, 20.0, 22.0, 25.0, 30.0]
    if V == 4096:
        boosts = [b - math.log(128256 / 4096) for b in boosts]
    cfg, cfg_o = lib_cfg(wl), oracle_cfg(wl)
    block = synth.peaked_draft_logits(wl, DEV, boosts, seed)[:, :, 0, :].contiguous()
    roots, L = synth.root_tokens(wl), synth.prefix_lengths(wl)
    s_np, _ = synth.zipf_M(wl.V, wl.W, seed)
    status = _status()
    gpu = gb().graft_build_tree(cfg, block, roots.to(DEV), torch.from_numpy(s_np).to(DEV), L.to(DEV), status=status,
                                block=True)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    trees, margins, fns = _oracle_tree(wl, cfg_o, block, roots, s_np, L, block=True)
    exact = _check_trees(gpu, trees, margins, fns, roots, s_np, L, cfg_o)
    assert exact >= wl.B - 2, f"too many near-tie requests: {margins}"


def test_build_tree_empty_M_pads_the_graft():
    """An all-empty M: pruned trees keep their draft nodes and every grafted slot is a pad (token 0, in
    the template's shape), as the oracle builds it."""
    wl = _peaked_wl(4096, 12, 6)
    boosts = [b - math.log(128256 / 4096) for b in [0.0, 10.0, 13.0, 14.0, 15.0, 16.0, 17.0, 18.0, 20.0, 22.0, 25.0,
                                                    30.0]]
    cfg, cfg_o = lib_cfg(wl), oracle_cfg(wl)
    dl = synth.peaked_draft_logits(wl, DEV, boosts, 6)
    roots, L = synth.root_tokens(wl), synth.prefix_lengths(wl)
    s_np, _ = synth.empty_M(wl.V, wl.W)
    gpu = _build(wl, cfg, dl, roots, torch.from_numpy(s_np).to(DEV), L)
    trees, margins, fns = _oracle_tree(wl, cfg_o, dl, roots, s_np, L)
    exact = _check_trees(gpu, trees, margins, fns, roots, s_np, L, cfg_o)
    assert exact >= wl.B - 2
    tok = to_np(gpu["tok"])
    for b in range(wl.B):
        assert (tok[b, trees[b].n_draft:] == 0).all()


@pytest.mark.parametrize("V,seed", [(4096, 1), (128256, 2)])  # the drafts of test_build_tree_all_stages
def test_build_tree_without_retrieval(V, seed):
    """The 'w/o retrieval' ablation (graft_config_no_retrieval: K_ret = 0 at every stage): at every
    pruning stage the draft takes the whole budget, slots a short pool cannot fill are empty nodes
    (token -1 under the root), and the trees equal the oracle's."""
    wl = _peaked_wl(V, 12, seed)
    boosts = [0.0, 10.0, 13.0, 14.0, 15.0, 16.0, 17.0, 18.0, 20.0, 22.0, 25.0, 30.0]
    if V == 4096:
        boosts = [b - math.log(128256 / 4096) for b in boosts]
    cfg = gb().graft_config_no_retrieval(lib_cfg(wl))
    cfg_o = oracle_cfg(wl, no_retrieval=True)
    assert cfg.as_dict()["K_draft"] == cfg_o["K_draft"] and cfg.n_tmpl == 0
    dl = synth.peaked_draft_logits(wl, DEV, boosts, seed)
    roots, L = synth.root_tokens(wl), synth.prefix_lengths(wl)
    s_np, _ = synth.zipf_M(wl.V, wl.W, seed)  # a full M that must not be read
    gpu = _build(wl, cfg, dl, roots, torch.from_numpy(s_np).to(DEV), L)
    trees, margins, fns = _oracle_tree(wl, cfg_o, dl, roots, s_np, L)
    exact = _check_trees(gpu, trees, margins, fns, roots, s_np, L, cfg_o)
    assert exact >= wl.B - 2, f"too many near-tie requests: {margins}"
    tok, stages = to_np(gpu["tok"]), to_np(gpu["stage"])
    assert {0, 1, 2, 3} <= set(stages.tolist())
    for b in range(wl.B):
        n_pool = wl.k + ([0, 1, 5, wl.D - 1][int(stages[b])]) * wl.k ** 2
        n_real = min(wl.Kmax - 1, n_pool)
        assert (tok[b, 1:1 + n_real] >= 0).all() and (tok[b, 1 + n_real:] == gb().EMPTY_TOKEN).all()
    assert (tok == gb().EMPTY_TOKEN).any()  # a d0 prune left empty slots


def test_empty_nodes_are_never_accepted_and_add_no_pair():
    """Empty nodes of the no-retrieval ablation: even when the target's argmax at the root is token 0 (the
    pad token a retrieval miss would carry), an empty node is not accepted, and the M update adds pairs only
    for real nodes."""
    wl = synth.WORKLOADS["tiny"].scaled(V=500)
    cfg = gb().graft_config_no_retrieval(lib_cfg(wl, tau=1.5))  # c_0 <= 1 < 1.5: always pruned at d0
    cfg_o = oracle_cfg(wl, tau=1.5, no_retrieval=True)
    dl = synth.draft_logits(wl, DEV)
    roots, L = synth.root_tokens(wl), synth.prefix_lengths(wl)
    s_np, c_np = synth.empty_M(wl.V, wl.W)
    gpu = _build(wl, cfg, dl, roots, torch.from_numpy(s_np).to(DEV), L)
    trees, _, _ = _oracle_tree(wl, cfg_o, dl, roots, s_np, L)
    _compare_tree(gpu, trees)
    tok, par, dep = (to_np(gpu[k]) for k in ("tok", "parent", "depth"))
    assert int(to_np(gpu["stage"])[0]) == 0 and (tok[0] == -1).sum() == wl.Kmax - 1 - wl.k
    tl = synth.target_logits(wl, DEV)
    t0 = 0 if 0 not in tok[0, 1:].tolist() else min(set(range(wl.V)) - set(tok[0].tolist()))
    tl[0, 0, t0] = tl[0, 0].max() + 5.0  # the root's argmax: token 0 unless a draft child carries it
    Lcap = wl.lcap()
    Q, Kc, Vc, Kt, Vt = synth.layer_tensors(wl, 0, DEV, Lcap=Lcap)
    ptr = lambda ts: gb().layer_pointers(ts, DEV)
    status = _status()
    out = gb().graft_accept_compact(tl, gpu["tok"], gpu["parent"], gpu["depth"], ptr([Kc]), ptr([Vc]), ptr([Kt]),
                                    ptr([Vt]), 1, wl.Hkv, Lcap, L.to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oacc.accept_batch(to_np(tl), dict(tok=tok, parent=par, depth=dep))
    for k in ("argmax", "acc_len", "path", "out_tok", "bonus"):
        assert np.array_equal(to_np(out[k]), ref[k]), k
    assert int(ref["argmax"][0, 0]) == t0 and int(ref["acc_len"][0]) == 1  # no empty node accepted
    Ms, Mc = torch.from_numpy(s_np).to(DEV), torch.from_numpy(c_np).to(DEV)
    status = _status()
    gb().graft_update_M(Ms, Mc, gpu["tok"].view(-1), out["argmax"].view(-1), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0  # empty nodes are skipped silently
    want_s, want_c = oupd.update_M(s_np, c_np, tok.reshape(-1), ref["argmax"].reshape(-1))
    assert np.array_equal(to_np(Ms), want_s) and np.array_equal(to_np(Mc), want_c)
    assert int(want_c.sum()) == 1 + wl.k
