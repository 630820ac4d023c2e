"""GPU parity of the prompt-evidence M policy: seeding from a prompt's bigrams and the per-step refresh
from the emitted tokens (graft_update_M_emitted)."""
import numpy as np
import pytest
import torch

from oracle import update_m as oupd
from tests.helpers import gb, to_np
from tree_verification_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _M(V, W, seed):
    s, c = synth.zipf_M(V, W, seed)
    return s, c


@pytest.mark.parametrize("V,W,n", [(300, 8, 5000), (128256, 16, 65536)])
def test_seed_from_prompt_bigrams(V, W, n):
    succ, cnt = oupd.empty_M(V, W)
    toks = synth.token_stream(n, V, 13)
    want_s, want_c = oupd.update_M(succ, cnt, toks[:-1], toks[1:])
    Ms, Mc = torch.from_numpy(succ).to(DEV), torch.from_numpy(cnt).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gb().graft_seed_M_from_tokens(Ms, Mc, torch.from_numpy(toks).to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(to_np(Ms), want_s) and np.array_equal(to_np(Mc), want_c)


@pytest.mark.parametrize("B,Kmax,V,W", [(1, 64, 5000, 16), (64, 64, 2000, 16), (5, 32, 400, 8)])
def test_update_from_emitted_tokens(B, Kmax, V, W):
    rng = np.random.default_rng(B * 7 + Kmax)
    succ, cnt = _M(V, W, B)
    tree_tok = rng.integers(0, V, (B, Kmax)).astype(np.int32)
    acc_len = rng.integers(1, 7, B).astype(np.int32)
    out_tok = np.full((B, Kmax), -1, np.int32)
    for b in range(B):
        # small vocabulary slice: repeated bigrams across requests exercise multiplicities
        out_tok[b, :acc_len[b]] = rng.integers(0, min(V, 50), acc_len[b])
    want_s, want_c = oupd.update_M(succ, cnt, *oupd.emitted_pairs(tree_tok, out_tok, acc_len))
    Ms, Mc = torch.from_numpy(succ).to(DEV), torch.from_numpy(cnt).to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    t = lambda a: torch.from_numpy(a).to(DEV)
    gb().graft_update_M_emitted(Ms, Mc, t(tree_tok), t(out_tok), t(acc_len), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(to_np(Ms), want_s) and np.array_equal(to_np(Mc), want_c)
