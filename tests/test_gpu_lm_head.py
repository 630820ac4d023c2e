"""GPU parity of graft_lm_head_argmax (fused lm_head argmax) and of acceptance from a given argmax."""
import numpy as np
import pytest
import torch

from oracle import accept as oacc
from oracle import lm_head as olm
from tests.helpers import gb, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
CERT = 1e-2  # rows whose two best float64 logits are closer than this may legitimately pick either


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


def _check_rows(H, W, got, got_max, rows=None):
    """Exact on certified rows, valid (within CERT of the best) elsewhere; max logit within fp32 rounding."""
    Hn = H.float().numpy() if rows is None else H.float().numpy()[rows]
    lg = olm.logits(Hn, W.float().numpy())
    g, mx = olm.argmax_rows(lg)
    mg = olm.margins(lg)
    got = got if rows is None else got[rows]
    got_max = got_max if rows is None else got_max[rows]
    cert = mg >= CERT
    assert np.array_equal(got[cert], g[cert])
    idx = np.arange(len(got))
    assert np.all(lg[idx, got] >= mx - CERT)
    assert np.all(np.abs(got_max - mx) <= 1e-4 * (1.0 + np.abs(mx)))
    return int(cert.sum())


@pytest.mark.parametrize("N,d,V", [
    (1, 8, 1),            # a single token and vocabulary entry
    (100, 256, 5000),     # ragged row and token tiles
    (129, 136, 257),      # hidden size not a multiple of the 64-wide k slice
    (64, 4096, 128256),   # the LLaMA-3-8B verify step's lm_head (B 1, Kmax 64)
])
def test_lm_head_argmax_parity(N, d, V):
    H, W = _bf16((N, d), 11 + N), _bf16((V, d), 17 + V)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    g, mx = gb().graft_lm_head_argmax(H.to(DEV), W.to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    n_cert = _check_rows(H, W, to_np(g), to_np(mx))
    assert n_cert >= 0.9 * N


def test_lm_head_argmax_ties_and_planted_full_size():
    """Batched Qwen3-8B-sized product (4096 rows, 151936 tokens, d 4096): planted rows W[t_n] = 4 H[n]
    make t_n each row's unique argmax (a property at any size); duplicate rows test ties; sampled
    rows are checked against the oracle."""
    N, d, V = 4096, 4096, 151936
    H = _bf16((N, d), 5)
    W = _bf16((V, d), 6)
    rng = np.random.default_rng(0)
    t = 2 * rng.choice((V - 1) // 2, N, replace=False)  # even ids: t + 1 is never another planted id
    W[torch.from_numpy(t)] = (H.float() * 4).to(torch.bfloat16)
    tie_rows = np.arange(8)
    W[torch.from_numpy(t[tie_rows] + 1)] = W[torch.from_numpy(t[tie_rows])]  # duplicate just above: tie
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    g, mx = gb().graft_lm_head_argmax(H.to(DEV), W.to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    g = to_np(g)
    assert np.array_equal(g, t.astype(np.int32))  # planted, ties to the lower id
    sample = np.array(list(range(8)) + list(rng.choice(N, 24, replace=False)))
    _check_rows(H, W, g, to_np(mx), rows=sample)


def test_accept_from_given_argmax():
    """graft_accept_compact with target_logits NULL and the fused argmax equals the oracle's acceptance."""
    B, Kmax, d, V, Hkv, Lcap = 3, 16, 128, 700, 2, 64
    rng = np.random.default_rng(4)
    H = _bf16((B * Kmax, d), 21)
    W = _bf16((V, d), 22)
    g, _ = gb().graft_lm_head_argmax(H.to(DEV), W.to(DEV))
    torch.cuda.synchronize()
    g_np = to_np(g).reshape(B, Kmax)
    parent = np.full((B, Kmax), -1, np.int32)
    depth = np.zeros((B, Kmax), np.int32)
    tok = np.zeros((B, Kmax), np.int32)
    for b in range(B):
        for i in range(1, Kmax):
            parent[b, i] = rng.integers(0, i)
            depth[b, i] = depth[b, parent[b, i]] + 1
            # accept about half the edges
            tok[b, i] = g_np[b, parent[b, i]] if rng.random() < 0.6 else rng.integers(0, V)
    t32 = lambda a: torch.from_numpy(a).to(DEV)
    Kc = torch.zeros(B, Lcap, Hkv, 128, dtype=torch.bfloat16, device=DEV)
    Vc = torch.zeros_like(Kc)
    Kt = torch.randn(B, Kmax, Hkv, 128, device=DEV).to(torch.bfloat16)
    Vt = torch.randn(B, Kmax, Hkv, 128, device=DEV).to(torch.bfloat16)
    ptrs = lambda t: gb().layer_pointers([t], DEV)
    L = torch.tensor([5, 0, 17], dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = gb().graft_accept_compact(None, t32(tok), t32(parent), t32(depth), ptrs(Kc), ptrs(Vc), ptrs(Kt), ptrs(Vt), 1,
                                    Hkv, Lcap, L, status=status, argmax=g.view(B, Kmax), V=V)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for b in range(B):
        _, n, path, out_tok, bonus = oacc.accept_from_argmax(g_np[b], tok[b], parent[b], depth[b])
        assert int(out["acc_len"][b]) == n
        assert to_np(out["path"][b])[:n].tolist() == path
        assert to_np(out["out_tok"][b])[:n].tolist() == out_tok
        assert int(out["bonus"][b]) == bonus
        L0 = [5, 0, 17][b]
        assert torch.equal(Kc[b, L0:L0 + n].cpu(), Kt[b, torch.tensor(path)].cpu())
    assert to_np(L).tolist() == [5 + int(out["acc_len"][0]), int(out["acc_len"][1]), 17 + int(out["acc_len"][2])]
