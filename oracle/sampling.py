"""Lossless sampling acceptance: the target's sample at every tree node (oracle, test infrastructure).

Graft article, architecture paragraph and Graft abstract: verification is
lossless, i.e. the emitted tokens follow the target's own distribution.  With
temperature T > 0 the target's distribution at a node is softmax(logits / T).
Every proposal in a Graft tree is deterministic (the drafter's top-k, the
retrieved successors), and for deterministic proposals the standard
speculative-sampling rule over a node's children -- try the children in
order, accept child i with probability p'(x_i), and on rejection remove x_i
from p' and renormalise -- accepts child i with probability p(x_i) and emits
from p otherwise.  The same law results from drawing ONE sample y ~ p per node
and accepting the first child whose token is y (the bonus token is y where no
child matches).  The oracle does the latter: the target's sample is
argmax_v(logits[v] / T + G_v) with Gumbel noise G (the Gumbel-max trick), and
acceptance is then the greedy rule applied to these samples.

Noise is keyed by (seed, request, position of the sampled token, token id)
through the counter-based generator Philox-4x32-10 (Salmon, Moraes, Dror and
Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC 2011).  Keying by
position makes tree decoding emit exactly what autoregressive sampling with
the same noise would, which tests/test_oracle_sampling.py checks on the tiny
model.  Counter (v // 4, position, request, 0), key (seed low, seed high)
32-bit words; output word v % 4 gives the 32-bit draw x, and
u = ((x >> 9) + 1/2) / 2^23 (24 significant bits: exact in float32, so both
sides start from the same u), G = -log(-log(u)).
"""
from __future__ import annotations

import numpy as np

M0, M1 = 0xD2511F53, 0xCD9E8D57      # Philox-4x32 round multipliers
W0, W1 = 0x9E3779B9, 0xBB67AE85      # Weyl key increments
MASK = 0xFFFFFFFF


def philox4x32_10(ctr, key):
    """Philox-4x32 with 10 rounds on uint32 arrays: ctr [..., 4], key [..., 2] -> [..., 4]."""
    c = [np.asarray(ctr[..., i], dtype=np.uint64) for i in range(4)]
    k0 = np.asarray(key[..., 0], dtype=np.uint64)
    k1 = np.asarray(key[..., 1], dtype=np.uint64)
    for r in range(10):
        p0 = np.uint64(M0) * c[0]
        p1 = np.uint64(M1) * c[2]
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(MASK)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(MASK)
        c = [(hi1 ^ c[1] ^ k0) & np.uint64(MASK), lo1, (hi0 ^ c[3] ^ k1) & np.uint64(MASK), lo0]
        if r < 9:
            k0 = (k0 + np.uint64(W0)) & np.uint64(MASK)
            k1 = (k1 + np.uint64(W1)) & np.uint64(MASK)
    return np.stack(c, axis=-1).astype(np.uint32)


def draws(seed: int, b: int, pos: int, V: int) -> np.ndarray:
    """The 32-bit draws x[v] for request b, sampled position pos, tokens v < V."""
    n4 = (V + 3) // 4
    ctr = np.zeros((n4, 4), np.uint32)
    ctr[:, 0] = np.arange(n4, dtype=np.uint32)
    ctr[:, 1] = np.uint32(pos & MASK)
    ctr[:, 2] = np.uint32(b & MASK)
    key = np.array([seed & MASK, (seed >> 32) & MASK], np.uint32)
    return philox4x32_10(ctr, np.broadcast_to(key, (n4, 2))).reshape(-1)[:V]


def uniforms(x: np.ndarray) -> np.ndarray:
    return ((x >> np.uint32(9)).astype(np.float64) + 0.5) / float(1 << 23)


def gumbel(seed: int, b: int, pos: int, V: int) -> np.ndarray:
    return -np.log(-np.log(uniforms(draws(seed, b, pos, V))))


def sample_row(logits: np.ndarray, T: float, seed: int, b: int, pos: int):
    """(sampled token, gap between the best and second-best perturbed score)."""
    z = np.asarray(logits, np.float64) / T + gumbel(seed, b, pos, len(logits))
    y = int(np.argmax(z))
    if len(z) < 2:
        return y, np.inf
    top2 = np.partition(z, -2)[-2:]
    return y, float(top2[1] - top2[0])


def sample_tree(logits: np.ndarray, tree_pos: np.ndarray, T: float, seed: int):
    """Samples [B][Kmax] for target logits [B][Kmax][V]; node i samples the token at tree_pos + 1."""
    B, K, _ = logits.shape
    y = np.zeros((B, K), np.int32)
    gap = np.zeros((B, K))
    for b in range(B):
        for i in range(K):
            y[b, i], gap[b, i] = sample_row(logits[b, i], T, seed, b, int(tree_pos[b, i]) + 1)
    return y, gap
