"""GPU parity of the sampling-acceptance kernels: the target's sample per node from given logits
(graft_sample_tokens) and fused into the lm_head product (graft_lm_head_sample)."""
import numpy as np
import pytest
import torch

from oracle import lm_head as olm
from oracle import sampling as osmp
from tests.helpers import gb, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
CERT = 1e-3  # perturbed scores closer than this may legitimately resolve either way (float32 vs float64)


def _check(logits, pos, T, seed, got):
    """Exact where the oracle's best perturbed score leads by CERT, valid (within CERT) elsewhere."""
    B, K, V = logits.shape
    want, gap = osmp.sample_tree(logits, pos, T, seed)
    cert = gap >= CERT
    assert np.array_equal(got[cert], want[cert])
    for b in range(B):
        for i in range(K):
            if not cert[b, i]:
                z = logits[b, i] / T + osmp.gumbel(seed, b, int(pos[b, i]) + 1, V)
                assert z[got[b, i]] >= z.max() - CERT
    return int(cert.sum())


@pytest.mark.parametrize("V,T,seed", [(5000, 1.0, 7), (5000, 0.5, (1 << 40) + 3), (128256, 2.0, 11), (3, 1.0, 5),
                                        (4097, 0.05, 13), (128256, 0.1, 17)])  # (low T: most noise skipped)
def test_sample_tokens_parity(V, T, seed):
    B, K = 3, 16
    rng = np.random.default_rng(seed & 0xFFFF)
    logits = (rng.normal(size=(B, K, V)) * 3).astype(np.float32)
    pos = (rng.integers(0, 5000, (B, 1)) + rng.integers(0, 8, (B, K))).astype(np.int32)
    got = gb().graft_sample_tokens(torch.from_numpy(logits).to(DEV), torch.from_numpy(pos).to(DEV), T, seed)
    torch.cuda.synchronize()
    n_cert = _check(logits, pos, T, seed, to_np(got))
    assert n_cert >= 0.9 * B * K


@pytest.mark.parametrize("V,d,T", [(3000, 256, 0.8), (20000, 256, 0.05), (20000, 256, 8.0), (5000, 1024, 1.0)])
def test_lm_head_sample_parity(V, d, T):
    """The fused sampler against the oracle's Gumbel-max at temperatures where most tokens cannot win
    (T 0.05: the kernel draws no noise for them) and where nearly all can (T 8), over many token
    tiles."""
    B, K, seed = 2, 24, 99
    g = torch.Generator().manual_seed(3)
    H = torch.randn(B * K, d, generator=g).to(torch.bfloat16)
    W = torch.randn(V, d, generator=g).to(torch.bfloat16)
    pos = (np.arange(K)[None, :] // 3 + np.array([[100], [7]])).astype(np.int32)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = gb().graft_lm_head_sample(H.to(DEV), W.to(DEV), torch.from_numpy(pos).to(DEV), T, seed, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    logits = olm.logits(H.float().numpy(), W.float().numpy()).reshape(B, K, V)
    n_cert = _check(logits, pos, T, seed, to_np(got).reshape(B, K))
    assert n_cert >= 0.9 * B * K


def test_verify_step_with_sampling_and_emitted_policy():
    """A whole step at temperature 0.7 with M refreshed from the tree pairs and the emitted bigrams,
    against the oracle run on the same inputs."""
    from oracle import accept as oacc
    from oracle import config as oconfig
    from oracle import tree as otree
    from oracle import update_m as oupd
    from tree_verification_gb300 import synth
    from tree_verification_gb300.step import VerifyStep

    wl = synth.WORKLOADS["tiny"]
    cfg = gb().graft_config_init(wl.Kmax, wl.D, wl.k, wl.V, wl.W, list(wl.checkpoints), wl.tau)
    cfg_o = oconfig.make_config(Kmax=wl.Kmax, D=wl.D, k=wl.k, V=wl.V, W=wl.W)
    Lcap = wl.lcap()
    dl = synth.draft_logits(wl, DEV)
    roots, L0 = synth.root_tokens(wl), synth.prefix_lengths(wl)
    s_np, c_np = synth.zipf_M(wl.V, wl.W, wl.seed + 5)
    Q, Kc, Vc, Kt, Vt = synth.layer_tensors(wl, 0, DEV, Lcap=Lcap)
    res = otree.draft_tree(lambda d, f, _p: dl[0, d, f].cpu().numpy(), int(roots[0]), cfg_o)
    tree = otree.merge(int(roots[0]), otree.retained_draft(res, cfg_o),
                       otree.retrieve(int(roots[0]), s_np, cfg_o["tmpl_parent"], cfg_o["tmpl_rank"]),
                       cfg_o["tmpl_parent"], res.stage, int(L0[0]), cfg_o)
    tl = synth.target_logits(wl, DEV) * 4.0  # peaked enough that sampling accepts a few nodes
    T, seed = 0.7, 5
    y, gap = osmp.sample_tree(tl.cpu().numpy(), np.array(tree.pos)[None], T, seed)
    assert gap.min() >= CERT
    g, n, path, out_tok, bonus = oacc.accept_from_argmax(y[0], tree.tok, tree.parent, tree.depth)
    succ, cnt = oupd.update_M(s_np, c_np, np.array(tree.tok), y[0])
    succ, cnt = oupd.update_M(succ, cnt, *oupd.emitted_pairs(np.array([tree.tok]), np.array([out_tok + [-1]]),
                                                            np.array([n])))
    M_succ, M_cnt = torch.from_numpy(s_np).to(DEV), torch.from_numpy(c_np).to(DEV)
    L = L0.to(DEV)
    step = VerifyStep(cfg, wl.B, wl.Hq, wl.Hkv, 1, Lcap, DEV, [Kc], [Vc], [Kt], [Vt], m_policy="both",
                      temperature=T, seed=seed)
    step.run(dl, roots.to(DEV), M_succ, M_cnt, L, [Q], tl)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    assert int(step.acc["acc_len"][0]) == n
    assert to_np(step.acc["out_tok"][0])[:n].tolist() == out_tok
    assert int(step.acc["bonus"][0]) == bonus
    assert np.array_equal(to_np(M_succ), succ) and np.array_equal(to_np(M_cnt), cnt)
