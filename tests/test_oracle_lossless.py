"""Losslessness pin: hybrid-tree greedy decoding equals autoregressive greedy (CPU only).

Graft article (architecture paragraph) and Graft abstract state the method is
lossless.  On a tiny random-init transformer the oracle's whole step (draft
with pruning, retrieval from M, merge, tree attention, acceptance, KV
compaction, M update) must emit exactly the autoregressive greedy tokens and
leave the same KV cache behind.
"""
import numpy as np
import pytest

from oracle import config, tiny_lm


@pytest.fixture(scope="module")
def lm():
    return tiny_lm.TinyLM(seed=0)


@pytest.mark.parametrize("sharpen,seed", [(1.0, 1), (8.0, 2), (0.5, 3)])
def test_hybrid_greedy_equals_autoregressive(lm, sharpen, seed):
    rng = np.random.default_rng(seed)
    # a prompt with a repeated segment gives retrieval something to find
    seg = rng.integers(0, lm.V, 5).tolist()
    prompt = rng.integers(0, lm.V, 6).tolist() + seg + seg
    n_new = 36
    cfg = config.make_config(Kmax=16, D=4, k=3, V=lm.V, W=4, tau=0.3)
    ar, cache_ar, L_ar, margins = tiny_lm.greedy_ar(lm, prompt, n_new, 200)
    assert min(margins) > 1e-6  # argmax decisions are far from float64 noise
    hy, cache_hy, L_hy, steps = tiny_lm.greedy_hybrid(lm, prompt, n_new, 200, cfg, sharpen=sharpen, seed=seed)
    assert hy == ar
    n = min(L_ar, L_hy)
    for ca, ch in zip(cache_ar, cache_hy):
        assert np.allclose(ca["K"][:n], ch["K"][:n], atol=1e-9, rtol=0)
        assert np.allclose(ca["V"][:n], ch["V"][:n], atol=1e-9, rtol=0)
    # the run really took multi-token steps
    assert max(s["acc_len"] for s in steps) > 1


def test_stages_and_retrieval_are_exercised(lm):
    """Across a few prompts every pruning stage occurs and retrieved nodes get accepted."""
    cfg = config.make_config(Kmax=16, D=4, k=3, V=lm.V, W=4, tau=0.3)
    seen_stages, retrieved = set(), 0
    for seed, sharpen in ((1, 0.3), (2, 1.0)):
        prompt = np.random.default_rng(seed).integers(0, lm.V, 12).tolist()
        ar, *_ = tiny_lm.greedy_ar(lm, prompt, 40, 200)
        hy, _, _, steps = tiny_lm.greedy_hybrid(lm, prompt, 40, 200, cfg, sharpen=sharpen, seed=seed)
        assert hy == ar
        seen_stages |= {s["stage"] for s in steps}
        retrieved += sum(s["retrieved_accepted"] for s in steps)
    assert seen_stages == {0, 1, 2}
    assert retrieved > 0


def test_without_retrieval_is_lossless(lm):
    """The 'w/o retrieval' ablation (K_ret = 0, empty slots where a pruned pool runs short) emits the
    autoregressive greedy tokens too, and its pruned steps really carry empty nodes."""
    cfg = config.make_config(Kmax=16, D=4, k=3, V=lm.V, W=4, tau=0.3, no_retrieval=True)
    empties, stages = 0, set()
    for seed, sharpen in ((1, 0.3), (4, 1.0)):
        prompt = np.random.default_rng(seed).integers(0, lm.V, 12).tolist()
        ar, *_ = tiny_lm.greedy_ar(lm, prompt, 30, 200)
        hy, _, _, steps = tiny_lm.greedy_hybrid(lm, prompt, 30, 200, cfg, sharpen=sharpen, seed=seed)
        assert hy == ar
        assert all(s["retrieved_accepted"] == 0 for s in steps)
        empties += sum(s["empty_nodes"] for s in steps)
        stages |= {s["stage"] for s in steps}
    assert empties > 0 and 0 in stages
