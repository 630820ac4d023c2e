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


@pytest.mark.parametrize("V,T,seed", [(5000, 1.0, 7), (5000, 0.5, (1 << 40) + 3), (128256, 2.0, 11), (3, 1.0, 5)])
def test_sample_tokens_parity(V, T, seed):
    B, K = 3, 16
    rng = np.random.default_rng(seed & 0xFFFF)
    logits = (rng.normal(size=(B, K, V)) * 3).astype(np.float32)
    pos = (rng.integers(0, 5000, (B, 1)) + rng.integers(0, 8, (B, K))).astype(np.int32)
    got = gb().graft_sample_tokens(torch.from_numpy(logits).to(DEV), torch.from_numpy(pos).to(DEV), T, seed)
    torch.cuda.synchronize()
    n_cert = _check(logits, pos, T, seed, to_np(got))
    assert n_cert >= 0.9 * B * K


def test_lm_head_sample_parity():
    B, K, d, V, T, seed = 2, 24, 256, 3000, 0.8, 99
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
