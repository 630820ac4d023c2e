"""Tree-masked GQA attention of the verify forward (oracle, test infrastructure).

Graft article, architecture paragraph: the hybrid tree is verified on the
ordinary tree-attention path in one target forward pass.  Graft abstract:
expansive draft trees cost VRAM bandwidth and compute, which is where this
step's time goes.

This is the softmax-attention definition written out in float64:

    O[b, i, h] = sum_j softmax_j(q . k_j * scale) v_j

over the keys j that node i may see: every prefix key 0 .. L_b - 1 of its
request (unmasked) and every tree node j whose bit is set in node i's
ancestor-or-self mask.  Query head h reads KV head h // (Hq / Hkv).

Readings: no rotary embedding is applied here (Q and K arrive already
rotated); the scale is a parameter (1 / sqrt(head_dim) in every workload).
"""
from __future__ import annotations

import numpy as np


def mask_matrix(mask_b: np.ndarray, Kmax: int) -> np.ndarray:
    """Boolean [Kmax][Kmax] matrix: entry (i, j) is bit j of node i's mask."""
    bits = np.asarray(mask_b, dtype=np.uint64)
    j = np.arange(Kmax, dtype=np.uint64)
    return ((bits[:, None] >> j[None, :]) & np.uint64(1)).astype(bool)


def tree_attention_one(Q_b: np.ndarray, Kc_b: np.ndarray, Vc_b: np.ndarray, Kt_b: np.ndarray,
                       Vt_b: np.ndarray, L_b: int, mask_b: np.ndarray, scale: float,
                       heads=None) -> np.ndarray:
    """Attention for one request.

    Q_b [Kmax][Hq][d], Kc_b/Vc_b [>=L_b][Hkv][d], Kt_b/Vt_b [Kmax][Hkv][d],
    mask_b [Kmax] ancestor bitmasks.  Returns float64 [Kmax][Hq][d]
    (only the listed ``heads`` are filled when given).
    """
    Kmax, Hq, d = Q_b.shape
    Hkv = Kt_b.shape[1]
    group = Hq // Hkv
    allowed = np.concatenate([np.ones((Kmax, L_b), bool), mask_matrix(mask_b, Kmax)], axis=1)
    out = np.zeros((Kmax, Hq, d), np.float64)
    for h in (range(Hq) if heads is None else heads):
        g = h // group
        keys = np.concatenate([Kc_b[:L_b, g].astype(np.float64), Kt_b[:, g].astype(np.float64)], axis=0)
        vals = np.concatenate([Vc_b[:L_b, g].astype(np.float64), Vt_b[:, g].astype(np.float64)], axis=0)
        s = (Q_b[:, h].astype(np.float64) @ keys.T) * scale
        s = np.where(allowed, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h] = p @ vals
    return out


def tree_attention(Q, Kc, Vc, Kt, Vt, L, mask, scale: float) -> np.ndarray:
    """Batched tree attention: Q [B][Kmax][Hq][d], Kc/Vc [B][Lcap][Hkv][d],
    Kt/Vt [B][Kmax][Hkv][d], L [B], mask [B][Kmax]; returns float64 O like Q."""
    B = Q.shape[0]
    return np.stack([tree_attention_one(Q[b], Kc[b], Vc[b], Kt[b], Vt[b], int(L[b]), mask[b], scale)
                     for b in range(B)])
