"""Seeded synthetic inputs for the verify step (shared by tests and the benchmark).

This module holds only input generation: random draws with fixed seeds and
the shapes, value distributions and structure of the five workloads below.
It contains none of the method's arithmetic.  The only structural helper,
``plant_paths``, edits target logits so that a chosen root path of a given
tree becomes the target's greedy continuation.

Workloads (sizes as the Graft pages' settings suggest; the pages' benchmark
datasets are replaced by these seeded draws):

* ``tiny``            batch 1, vocab 32000, M 32000x8 with Zipf(1.1) counts,
                      draft depth 6 top-4, logits N(0, 2), tau 0.3, Kmax 32,
                      1 layer, 8/2 heads, prefix 512, planted path length 5
* ``llama3_8b``       batch 1, 32/8 heads, 32 layers, prefix 4096, Kmax 64,
                      depth 8 top-8, vocab 128256, M 128256x16 (starts empty),
                      planted path length 5
* ``qwen3_8b_batch``  batch 64, 32/8 heads, prefixes uniform in [512, 4096],
                      Kmax 64, vocab 151936, M 151936x16 shared and updated
                      from all trees, planted lengths uniform in [1, 6];
                      36 layers (the Qwen3-8B depth, not stated on the pages)
* ``llama31_8b_long`` batch 1, prefix 65536, 32/8 heads, 32 layers, Kmax 64,
                      vocab 128256, M pre-warmed by 5 updates with every
                      adjacent pair of a seeded 65536-token stream
* ``qwen3_235b``      batch 16, 64/4 heads, 94 layers, prefix 8192, Kmax 64,
                      vocab 151936, M 151936x32 updated per step, planted
                      lengths uniform in [1, 7]

Activations and KV are bf16 N(0, 1); target logits are fp32 N(0, 1).
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    n_layers: int
    L: Tuple[int, int]          # prefix length range [lo, hi] (lo == hi: fixed)
    Kmax: int
    D: int
    k: int
    V: int
    W: int
    plant: Tuple[int, int]      # planted accepted-length range [lo, hi]
    M_init: str                 # "zipf", "empty" or "warm"
    tau: float = 0.3
    checkpoints: Tuple[int, ...] = (0, 1, 5)
    head_dim: int = 128
    seed: int = 0
    d_model: int = 4096         # hidden size of the target's final layer (lm_head input)

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv

    @property
    def Lmax(self) -> int:
        return self.L[1]

    def lcap(self, steps: int = 1) -> int:
        """Cache capacity for ``steps`` steps of growth, rounded up to 64 rows."""
        c = self.Lmax + steps * self.Kmax
        return (c + 63) // 64 * 64

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", B=1, Hq=8, Hkv=2, n_layers=1, L=(512, 512), Kmax=32, D=6, k=4, V=32000, W=8,
                     plant=(5, 5), M_init="zipf", d_model=256),
    "llama3_8b": Workload("llama3_8b", B=1, Hq=32, Hkv=8, n_layers=32, L=(4096, 4096), Kmax=64, D=8, k=8,
                          V=128256, W=16, plant=(5, 5), M_init="empty"),
    "qwen3_8b_batch": Workload("qwen3_8b_batch", B=64, Hq=32, Hkv=8, n_layers=36, L=(512, 4096), Kmax=64, D=8,
                               k=8, V=151936, W=16, plant=(1, 6), M_init="empty"),
    "llama31_8b_long": Workload("llama31_8b_long", B=1, Hq=32, Hkv=8, n_layers=32, L=(65536, 65536), Kmax=64, D=8,
                                k=8, V=128256, W=16, plant=(5, 5), M_init="warm"),
    "qwen3_235b": Workload("qwen3_235b", B=16, Hq=64, Hkv=4, n_layers=94, L=(8192, 8192), Kmax=64, D=8, k=8,
                           V=151936, W=32, plant=(1, 7), M_init="empty"),
}


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal(shape, std: float, seed: int, device, dtype=torch.float32) -> torch.Tensor:
    """N(0, std^2) draws of the given dtype (drawn in fp32, then cast)."""
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, std, generator=generator(seed, device))
    return t if dtype == torch.float32 else t.to(dtype)


def prefix_lengths(wl: Workload) -> torch.Tensor:
    lo, hi = wl.L
    if lo == hi:
        return torch.full((wl.B,), lo, dtype=torch.int32)
    rng = np.random.default_rng(wl.seed + 11)
    return torch.from_numpy(rng.integers(lo, hi + 1, wl.B).astype(np.int32))


def planted_lengths(wl: Workload) -> List[int]:
    lo, hi = wl.plant
    rng = np.random.default_rng(wl.seed + 13)
    return rng.integers(lo, hi + 1, wl.B).tolist()


def root_tokens(wl: Workload) -> torch.Tensor:
    rng = np.random.default_rng(wl.seed + 17)
    return torch.from_numpy(rng.integers(0, wl.V, wl.B).astype(np.int32))


def draft_logits(wl: Workload, device, std: float = 2.0) -> torch.Tensor:
    """[B][D][k][V] fp32 N(0, std^2)."""
    return normal((wl.B, wl.D, wl.k, wl.V), std, wl.seed + 19, device)


def peaked_draft_logits(wl: Workload, device, boosts: Sequence[float], seed: int = 0) -> torch.Tensor:
    """Drafter rows with a few dominant tokens, so the draft is confident.

    Row (b, d, f) is N(0, 2^2) plus boosts[b] on one random token and
    boosts[b] - 1.5 and boosts[b] - 3 on two more; larger boosts keep the
    confidence above the thresholds for more checkpoints.
    """
    x = normal((wl.B, wl.D, wl.k, wl.V), 2.0, wl.seed + 23 + seed, device)
    rng = np.random.default_rng(wl.seed + 29 + seed)
    for b in range(wl.B):
        ids = rng.integers(0, wl.V, (wl.D, wl.k, 3))
        for j, delta in enumerate((0.0, -1.5, -3.0)):
            idx = torch.from_numpy(ids[:, :, j]).to(device).long().unsqueeze(-1)
            x[b].scatter_add_(-1, idx, torch.full(idx.shape, float(boosts[b]) + delta, device=device))
    return x


def target_logits(wl: Workload, device) -> torch.Tensor:
    """[B][Kmax][V] fp32 N(0, 1)."""
    return normal((wl.B, wl.Kmax, wl.V), 1.0, wl.seed + 31, device)


def layer_tensors(wl: Workload, layer: int, device, Lcap: Optional[int] = None):
    """Q [B][Kmax][Hq][128], Kc/Vc [B][Lcap][Hkv][128], Kt/Vt [B][Kmax][Hkv][128], all bf16 N(0, 1)."""
    Lcap = wl.lcap() if Lcap is None else Lcap
    s = wl.seed * 7919 + 1000 * (layer + 1)
    d = wl.head_dim
    Q = normal((wl.B, wl.Kmax, wl.Hq, d), 1.0, s + 1, device, torch.bfloat16)
    Kc = normal((wl.B, Lcap, wl.Hkv, d), 1.0, s + 2, device, torch.bfloat16)
    Vc = normal((wl.B, Lcap, wl.Hkv, d), 1.0, s + 3, device, torch.bfloat16)
    Kt = normal((wl.B, wl.Kmax, wl.Hkv, d), 1.0, s + 4, device, torch.bfloat16)
    Vt = normal((wl.B, wl.Kmax, wl.Hkv, d), 1.0, s + 5, device, torch.bfloat16)
    return Q, Kc, Vc, Kt, Vt


def zipf_M(V: int, W: int, seed: int, a: float = 1.1, cap: int = 1 << 20):
    """M with W distinct uniform successors per row and Zipf(a) counts clamped to cap.

    Rows are stored in the table's ranked order (count desc, token asc).
    """
    rng = np.random.default_rng(seed)
    succ = rng.integers(0, V, (V, W))
    while True:  # resample duplicates within a row
        s = np.sort(succ, axis=1)
        dup_rows = np.nonzero((s[:, 1:] == s[:, :-1]).any(axis=1))[0]
        if dup_rows.size == 0:
            break
        succ[dup_rows] = rng.integers(0, V, (dup_rows.size, W))
    cnt = np.minimum(rng.zipf(a, (V, W)), cap)
    order = np.lexsort((succ, -cnt), axis=1)
    succ = np.take_along_axis(succ, order, axis=1).astype(np.int32)
    cnt = np.take_along_axis(cnt, order, axis=1).astype(np.int32)
    return succ, cnt


def empty_M(V: int, W: int):
    return np.full((V, W), -1, np.int32), np.zeros((V, W), np.int32)


def token_stream(n: int, V: int, seed: int) -> np.ndarray:
    """A uniform seeded token stream (the long-context prompt)."""
    return np.random.default_rng(seed).integers(0, V, n).astype(np.int32)


def stream_pairs(stream: np.ndarray):
    """All adjacent (src, dst) pairs of a token stream."""
    return stream[:-1].copy(), stream[1:].copy()


def plant_paths(logits: torch.Tensor, tok, parent, depth, lengths: Sequence[int]) -> List[int]:
    """Make a root path of the requested length the target's greedy continuation.

    For request b the end node is the lowest-index node of depth
    lengths[b] - 1, or the lowest-index deepest node when the tree is
    shallower.  Every edge parent -> child on its root path gets
    logits[b][parent][token(child)] = row max + 1; at the end node, if the
    row's argmax is one of its children's tokens, another token (the lowest
    id that is not a child token) is raised above it.  Duplicate paths may
    still extend acceptance; the reference decides.  Edits ``logits`` in
    place; returns the chosen end nodes.
    """
    tok = np.asarray(tok)
    parent = np.asarray(parent)
    depth = np.asarray(depth)
    B, K = tok.shape
    ends = []
    for b in range(B):
        want = max(1, int(lengths[b])) - 1
        dep = depth[b]
        cands = np.nonzero(dep == want)[0]
        if cands.size == 0:
            cands = np.nonzero(dep == dep.max())[0]
        end = int(cands[0])
        ends.append(end)
        j = end
        while j > 0:
            p = int(parent[b, j])
            row = logits[b, p]
            row[int(tok[b, j])] = row.max() + 1.0
            j = p
        children = {int(tok[b, c]) for c in range(K) if parent[b, c] == end}
        row = logits[b, end]
        if int(torch.argmax(row)) in children:
            t = 0
            while t in children:
                t += 1
            row[t] = row.max() + 1.0
    return ends


def lm_head_inputs(wl: Workload, device, seed_offset: int = 71):
    """Synthetic final hidden states [B*Kmax][d_model] and output embedding [V][d_model], bf16 N(0,1)."""
    g = torch.Generator(device="cpu").manual_seed(wl.seed + seed_offset)
    H = torch.randn(wl.B * wl.Kmax, wl.d_model, generator=g).to(torch.bfloat16).to(device)
    W = torch.randn(wl.V, wl.d_model, generator=g).to(torch.bfloat16).to(device)
    return H, W
