"""The whole GPU step, chained, against the oracle's whole step.

Graft article, architecture paragraph: one verify forward over the merged
tree, then acceptance, compaction and the online update of M.  Every other
GPU test feeds one stage inputs built by the oracle; here the GPU step runs
as a user runs it (VerifyStep: GPU tree -> GPU mask -> GPU attention -> GPU
acceptance and compaction -> GPU M update) for two consecutive steps, the
second starting from the first one's bonus token, lengths, caches and M, and
after each step every output is compared with oracle.step.verify_step run on
host copies of the same inputs:

* tree (tokens, parents, depths, positions, masks, stage), target argmax,
  accepted length, path, emitted tokens, bonus, new lengths, the whole KV
  caches of every layer and the table M: bit-exact;
* attention of the last layer on sampled requests, among them the longest
  and the shortest ones (the longest-first schedule runs those last), within
  the attention tolerance.

Workloads are the four large configurations with their full sizes (batch,
heads, prefix lengths, vocabulary, M) and the layer count cut to two.
Drafter logits whose decisions come within MARGIN of a tie are redrawn with
the next seed (seed + 1000 k), so every integer decision is certified.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from oracle import step as ostep
from oracle import tree as otree
from tests.helpers import MARGIN, assert_attention_close, gb, initial_M, lib_cfg, oracle_cfg, to_np
from tree_verification_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
N_LAYERS = 2


def _bits(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit words of a bf16 tensor (compaction is compared byte for byte)."""
    return t.view(torch.int16).cpu().numpy()


def _certified_drafts(wl, step, roots):
    """Drafter logits for this step whose tree decisions all clear MARGIN (redrawn otherwise)."""
    cfg_o = oracle_cfg(wl)
    for attempt in range(8):
        seed = wl.seed + 100 * (step + 1) + 1000 * attempt
        dl = synth.draft_logits(wl.scaled(seed=seed), DEV)
        ok = True
        for b in range(wl.B):
            rows = {}

            def row_fn(d, f, _p, b=b, rows=rows):
                if (d, f) not in rows:
                    rows[(d, f)] = dl[b, d, f].cpu().numpy()
                return rows[(d, f)]

            if otree.draft_margins(row_fn, int(roots[b]), cfg_o) <= MARGIN:
                ok = False
                break
        if ok:
            return dl, seed
    pytest.fail("no certified drafter logits in 8 draws")


def _sampled_requests(L0):
    order = np.lexsort((np.arange(len(L0)), -np.asarray(L0)))  # longest first, ties to the lower index
    picks = [int(order[0]), int(order[len(order) // 2])] + [int(x) for x in order[-2:]]
    return sorted(set(picks))


@pytest.mark.parametrize("name", ["llama3_8b", "qwen3_8b_batch", "llama31_8b_long", "qwen3_235b"])
def test_chained_step_matches_oracle(name):
    from tree_verification_gb300.step import VerifyStep

    wl = synth.WORKLOADS[name].scaled(n_layers=N_LAYERS)
    cfg, cfg_o = lib_cfg(wl), oracle_cfg(wl)
    Lcap = wl.lcap(2)  # room for two steps of growth
    scale = 1 / math.sqrt(128)
    s_np, c_np = initial_M(wl)
    Ms, Mc = torch.from_numpy(s_np).to(DEV), torch.from_numpy(c_np).to(DEV)
    L0 = synth.prefix_lengths(wl)
    layers = [synth.layer_tensors(wl, l, DEV, Lcap=Lcap) for l in range(N_LAYERS)]
    Kc = [x[1] for x in layers]
    Vc = [x[2] for x in layers]
    Kt = [x[3] for x in layers]
    Vt = [x[4] for x in layers]
    Q = [x[0] for x in layers]
    step = VerifyStep(cfg, wl.B, wl.Hq, wl.Hkv, N_LAYERS, Lcap, DEV, Kc, Vc, Kt, Vt)
    # host state the oracle carries from step to step
    Kc_h, Vc_h = [_bits(x) for x in Kc], [_bits(x) for x in Vc]
    L_h = L0.numpy().astype(np.int64)
    L = L0.to(DEV)
    roots = synth.root_tokens(wl)
    sampled = _sampled_requests(L0.numpy())
    for s in range(2):
        if s == 1:  # fresh queries and tree KV for the second step, written into the step's buffers
            for l in range(N_LAYERS):
                q2, _, _, kt2, vt2 = synth.layer_tensors(wl.scaled(seed=wl.seed + 7), l, DEV, Lcap=8)
                Q[l].copy_(q2)
                Kt[l].copy_(kt2)
                Vt[l].copy_(vt2)
        dl, _ = _certified_drafts(wl, s, roots)
        dl_h = dl.cpu().numpy()
        tree_o = otree.build_tree_batch(dl_h, roots.numpy(), s_np, L_h, cfg_o)
        tl = synth.target_logits(wl.scaled(seed=wl.seed + 50 * s), DEV)
        synth.plant_paths(tl, tree_o["tok"], tree_o["parent"], tree_o["depth"], synth.planted_lengths(wl))
        tl_h = tl.cpu().numpy()
        Q_h = [to_np(x) for x in Q]
        Kt_h, Vt_h = [_bits(x) for x in Kt], [_bits(x) for x in Vt]
        # attention reference of the last layer on the sampled requests (before compaction)
        ref_o = {}
        for b in sampled:
            lb = int(L_h[b])
            kc = torch.from_numpy(Kc_h[-1][b, :lb]).view(torch.bfloat16).float().numpy()
            vc = torch.from_numpy(Vc_h[-1][b, :lb]).view(torch.bfloat16).float().numpy()
            ref_o[b] = oatt.tree_attention_one(Q_h[-1][b], kc, vc, to_np(Kt[-1][b]), to_np(Vt[-1][b]), lb,
                                               tree_o["mask"][b], scale)

        step.run(dl, roots.to(DEV), Ms, Mc, L, Q, tl)
        torch.cuda.synchronize()
        assert int(step.status.item()) == 0

        # the oracle's whole step on the host copies (attention compared separately above)
        out = ostep.verify_step(cfg_o, dl_h, roots.numpy(), s_np, c_np, L_h, Q_h, Kc_h, Vc_h, Kt_h, Vt_h, tl_h,
                                scale, attn_layers=[])
        t = out["tree"]
        for k in ("tok", "parent", "depth", "pos", "stage"):
            assert np.array_equal(to_np(step.tree[k]), t[k]), f"step {s}: tree {k}"
        assert np.array_equal(step.tree["mask"].cpu().numpy().view(np.uint64), t["mask"]), f"step {s}: mask"
        a = out["accept"]
        for k in ("argmax", "acc_len", "path", "out_tok", "bonus"):
            assert np.array_equal(to_np(step.acc[k]), a[k]), f"step {s}: {k}"
        assert np.array_equal(to_np(L), out["L"]), f"step {s}: lengths"
        assert np.array_equal(to_np(Ms), out["M_succ"]) and np.array_equal(to_np(Mc), out["M_cnt"]), f"step {s}: M"
        for l in range(N_LAYERS):
            assert np.array_equal(_bits(Kc[l]), Kc_h[l]) and np.array_equal(_bits(Vc[l]), Vc_h[l]), \
                f"step {s}: cache of layer {l}"
        O = to_np(step.O)
        for b in sampled:
            assert_attention_close(O[b], ref_o[b])
        if name == "qwen3_8b_batch":
            assert len(set(a["acc_len"].tolist())) > 2  # planted lengths vary across the batch
        # carry the state into the next step
        s_np, c_np = out["M_succ"], out["M_cnt"]
        L_h = out["L"].astype(np.int64)
        roots = torch.from_numpy(a["bonus"].astype(np.int32))
        del dl, tl, dl_h, tl_h
        torch.cuda.empty_cache()
