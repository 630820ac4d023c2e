"""Pins for the oracle's tree attention against torch's scaled_dot_product_attention (CPU, fp64)."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as att


def _sdpa(q, k, v, allowed, scale):
    """Library reference: q [Hq][n][d], k/v [Hkv][m][d] expanded to Hq heads, allowed [n][m]."""
    group = q.shape[0] // k.shape[0]
    k = k.repeat_interleave(group, dim=0)
    v = v.repeat_interleave(group, dim=0)
    return F.scaled_dot_product_attention(q, k, v, attn_mask=allowed, scale=scale)


def _rand(shape, rng):
    return rng.normal(0, 1, shape)


@pytest.mark.parametrize("Hq,Hkv,K,d", [(4, 2, 8, 16), (8, 2, 5, 32), (4, 4, 3, 8)])
def test_chain_tree_equals_causal_attention(Hq, Hkv, K, d):
    rng = np.random.default_rng(Hq * 100 + K)
    Q = _rand((1, K, Hq, d), rng)
    Kt = _rand((1, K, Hkv, d), rng)
    Vt = _rand((1, K, Hkv, d), rng)
    empty = np.zeros((1, 4, Hkv, d))
    mask = np.array([[(1 << (i + 1)) - 1 for i in range(K)]], dtype=np.uint64)
    out = att.tree_attention(Q, empty, empty, Kt, Vt, np.array([0]), mask, 0.37)
    q = torch.from_numpy(Q[0]).permute(1, 0, 2)
    k = torch.from_numpy(Kt[0]).permute(1, 0, 2)
    v = torch.from_numpy(Vt[0]).permute(1, 0, 2)
    group = Hq // Hkv
    ref = F.scaled_dot_product_attention(q, k.repeat_interleave(group, 0), v.repeat_interleave(group, 0),
                                         is_causal=True, scale=0.37)
    assert np.allclose(out[0], ref.permute(1, 0, 2).numpy(), atol=1e-12, rtol=1e-12)


def test_prefix_plus_tree_equals_masked_sdpa():
    rng = np.random.default_rng(7)
    B, K, Hq, Hkv, d, Lcap = 2, 6, 8, 2, 16, 40
    L = np.array([33, 0])
    parent = [-1, 0, 0, 1, 1, 2]
    mask = []
    for i in range(K):
        mask.append((1 << i) | (mask[parent[i]] if parent[i] >= 0 else 0))
    masks = np.array([mask, mask], dtype=np.uint64)
    Q = _rand((B, K, Hq, d), rng)
    Kc, Vc = _rand((B, Lcap, Hkv, d), rng), _rand((B, Lcap, Hkv, d), rng)
    Kt, Vt = _rand((B, K, Hkv, d), rng), _rand((B, K, Hkv, d), rng)
    out = att.tree_attention(Q, Kc, Vc, Kt, Vt, L, masks, 1 / np.sqrt(d))
    for b in range(B):
        allowed = np.zeros((K, L[b] + K), bool)
        allowed[:, : L[b]] = True
        for i in range(K):
            j = i
            while j >= 0:
                allowed[i, L[b] + j] = True
                j = parent[j]
        keys = torch.from_numpy(np.concatenate([Kc[b, : L[b]], Kt[b]])).permute(1, 0, 2)
        vals = torch.from_numpy(np.concatenate([Vc[b, : L[b]], Vt[b]])).permute(1, 0, 2)
        ref = _sdpa(torch.from_numpy(Q[b]).permute(1, 0, 2), keys, vals, torch.from_numpy(allowed), 1 / np.sqrt(d))
        assert np.allclose(out[b], ref.permute(1, 0, 2).numpy(), atol=1e-12, rtol=1e-12)


def test_single_node_tree_is_decode_attention():
    """Kmax = 1: the root attends to the whole prefix plus itself, i.e. plain decode attention."""
    rng = np.random.default_rng(11)
    Hq, Hkv, d, L = 8, 2, 32, 50
    Q = _rand((1, 1, Hq, d), rng)
    Kc, Vc = _rand((1, L, Hkv, d), rng), _rand((1, L, Hkv, d), rng)
    Kt, Vt = _rand((1, 1, Hkv, d), rng), _rand((1, 1, Hkv, d), rng)
    out = att.tree_attention(Q, Kc, Vc, Kt, Vt, np.array([L]), np.array([[1]], np.uint64), 0.2)
    keys = torch.from_numpy(np.concatenate([Kc[0], Kt[0]])).permute(1, 0, 2)
    vals = torch.from_numpy(np.concatenate([Vc[0], Vt[0]])).permute(1, 0, 2)
    ref = _sdpa(torch.from_numpy(Q[0]).permute(1, 0, 2), keys, vals, None, 0.2)
    assert np.allclose(out[0], ref.permute(1, 0, 2).numpy(), atol=1e-12, rtol=1e-12)


def test_keys_past_length_are_ignored():
    rng = np.random.default_rng(5)
    Q = _rand((1, 2, 2, 8), rng)
    Kc, Vc = _rand((1, 10, 1, 8), rng), _rand((1, 10, 1, 8), rng)
    Kt, Vt = _rand((1, 2, 1, 8), rng), _rand((1, 2, 1, 8), rng)
    m = np.array([[1, 3]], np.uint64)
    a = att.tree_attention(Q, Kc, Vc, Kt, Vt, np.array([4]), m, 0.3)
    Kc[0, 4:] = 1e6
    Vc[0, 4:] = np.nan
    b = att.tree_attention(Q, Kc, Vc, Kt, Vt, np.array([4]), m, 0.3)
    assert np.array_equal(a, b)
