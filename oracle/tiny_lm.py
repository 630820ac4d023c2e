"""A tiny random-init transformer for the losslessness pin (oracle, test infrastructure).

Graft article, architecture paragraph, and Graft abstract: the method is
lossless, so hybrid-tree greedy decoding must emit exactly the tokens plain
autoregressive greedy decoding emits.  This module provides a small
float64 transformer (2 layers, d = 256, vocabulary 4096, GQA with rotary
positions) and both decoders; the hybrid decoder runs the oracle's tree
build, tree attention, acceptance, compaction and M update.

The draft model is outside the method's hot path (its weights are trained);
the hybrid decoder here drafts from the target's own logits, sharpened and
perturbed by seeded noise, which is enough to exercise every pruning stage.
"""
from __future__ import annotations

import math
from typing import List

import numpy as np

from . import accept as acc
from . import sampling as smp
from . import attention as att
from . import tree as tr
from . import update_m as um


class TinyLM:
    def __init__(self, V: int = 4096, d: int = 256, n_layers: int = 2, Hq: int = 4, Hkv: int = 2,
                 head_dim: int = 64, seed: int = 0):
        rng = np.random.default_rng(seed)
        self.V, self.d, self.Hq, self.Hkv, self.hd = V, d, Hq, Hkv, head_dim
        self.emb = rng.normal(0.0, 1.0, (V, d))
        self.layers = []
        for _ in range(n_layers):
            self.layers.append(dict(
                Wq=rng.normal(0.0, 1.0 / math.sqrt(d), (d, Hq * head_dim)),
                Wk=rng.normal(0.0, 1.0 / math.sqrt(d), (d, Hkv * head_dim)),
                Wv=rng.normal(0.0, 1.0 / math.sqrt(d), (d, Hkv * head_dim)),
                Wo=rng.normal(0.0, 1.0 / math.sqrt(Hq * head_dim), (Hq * head_dim, d)),
                W1=rng.normal(0.0, 1.0 / math.sqrt(d), (d, 4 * d)),
                W2=rng.normal(0.0, 1.0 / math.sqrt(4 * d), (4 * d, d))))
        self.Wlm = rng.normal(0.0, 3.0 / math.sqrt(d), (d, V))

    def new_cache(self, Lcap: int):
        return [dict(K=np.zeros((Lcap, self.Hkv, self.hd)), V=np.zeros((Lcap, self.Hkv, self.hd)))
                for _ in self.layers]

    @staticmethod
    def _rmsnorm(x):
        return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + 1e-6)

    def _rope(self, x, pos):
        half = self.hd // 2
        inv = 10000.0 ** (-np.arange(half) * 2.0 / self.hd)
        ang = np.asarray(pos, np.float64)[:, None] * inv[None, :]
        c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
        x0, x1 = x[..., 0::2], x[..., 1::2]
        out = np.empty_like(x)
        out[..., 0::2] = x0 * c - x1 * s
        out[..., 1::2] = x0 * s + x1 * c
        return out

    def forward(self, tokens, pos, mask, cache, L: int):
        """Run new tokens against a cache of length L.

        tokens/pos [n]; mask [n] ancestor-or-self bitmasks over the n new
        tokens.  Returns (logits [n][V], per-layer (K, V) of the new tokens).
        The cache is read, never written.
        """
        n = len(tokens)
        x = self.emb[np.asarray(tokens)]
        kv = []
        for lay, c in zip(self.layers, cache):
            h = self._rmsnorm(x)
            q = self._rope((h @ lay["Wq"]).reshape(n, self.Hq, self.hd), pos)
            k = self._rope((h @ lay["Wk"]).reshape(n, self.Hkv, self.hd), pos)
            v = (h @ lay["Wv"]).reshape(n, self.Hkv, self.hd)
            o = att.tree_attention_one(q, c["K"], c["V"], k, v, L, np.asarray(mask, np.uint64),
                                       1.0 / math.sqrt(self.hd))
            x = x + o.reshape(n, -1) @ lay["Wo"]
            h = self._rmsnorm(x)
            u = h @ lay["W1"]
            x = x + (u / (1.0 + np.exp(-u))) @ lay["W2"]
            kv.append((k, v))
        return self._rmsnorm(x) @ self.Wlm, kv


def greedy_ar(lm: TinyLM, prompt: List[int], n_new: int, Lcap: int):
    """Plain autoregressive greedy decoding; returns (tokens, cache, L, top-2 margins)."""
    cache = lm.new_cache(Lcap)
    L = 0
    logits = None
    out: List[int] = []
    margins: List[float] = []

    def push(tok):
        nonlocal L, logits
        lg, kv = lm.forward([tok], [L], [1], cache, L)
        for c, (k, v) in zip(cache, kv):
            c["K"][L] = k[0]
            c["V"][L] = v[0]
        L += 1
        logits = lg[0]

    for t in prompt:
        push(t)
    while len(out) < n_new:
        srt = np.sort(logits)
        margins.append(float(srt[-1] - srt[-2]))
        g = int(np.argmax(logits))
        out.append(g)
        push(g)
    return out, cache, L, margins


def greedy_hybrid(lm: TinyLM, prompt: List[int], n_new: int, Lcap: int, cfg: dict,
                  sharpen: float = 8.0, noise: float = 1.0, seed: int = 0):
    """Hybrid-tree greedy decoding with the oracle's stages.

    Returns (tokens, cache, L, per-step records).  M starts empty and is
    updated from every verified tree.
    """
    rng = np.random.default_rng(seed)
    cache = lm.new_cache(Lcap)
    L = 0
    for t in prompt[:-1]:
        _, kv = lm.forward([t], [L], [1], cache, L)
        for c, (k, v) in zip(cache, kv):
            c["K"][L] = k[0]
            c["V"][L] = v[0]
        L += 1
    root = prompt[-1]
    M_succ, M_cnt = um.empty_M(lm.V, cfg["W"])
    out: List[int] = []
    steps = []
    while len(out) < n_new:
        def row_fn(d, f, path, L=L):
            chain = [(1 << (i + 1)) - 1 for i in range(len(path))]
            lg, _ = lm.forward(path, [L + i for i in range(len(path))], chain, cache, L)
            return (sharpen * lg[-1] + rng.normal(0.0, noise, lm.V)).astype(np.float32)

        res = tr.draft_tree(row_fn, root, cfg)
        nodes = tr.retained_draft(res, cfg)
        ret = tr.retrieve(root, M_succ, cfg["tmpl_parent"], cfg["tmpl_rank"])
        tree = tr.merge(root, nodes, ret, cfg["tmpl_parent"], res.stage, L, cfg)
        # an empty node (token -1) runs through the model as token 0; it is never accepted
        logits, kv = lm.forward([max(t, 0) for t in tree.tok], tree.pos, tree.mask, cache, L)
        g, n, path, out_tok, bonus = acc.accept(logits, tree.tok, tree.parent, tree.depth)
        for c, (k, v) in zip(cache, kv):
            for t, p in enumerate(path):
                c["K"][L + t] = k[p]
                c["V"][L + t] = v[p]
        L += n
        out.extend(out_tok)
        root = bonus
        M_succ, M_cnt = um.update_M(M_succ, M_cnt, np.array(tree.tok), np.array(g))
        steps.append(dict(stage=res.stage, acc_len=n,
                          retrieved_accepted=sum(1 for p in path if p >= tree.n_draft),
                          empty_nodes=sum(1 for t in tree.tok if t == tr.EMPTY)))
    return out[:n_new], cache, L, steps


def sample_ar(lm: TinyLM, prompt: List[int], n_new: int, Lcap: int, T: float, seed: int):
    """Autoregressive sampling at temperature T with the position-keyed Gumbel noise of
    oracle.sampling; returns (tokens, cache, L, perturbed-score gaps)."""
    cache = lm.new_cache(Lcap)
    L = 0
    logits = None
    out: List[int] = []
    gaps: List[float] = []

    def push(tok):
        nonlocal L, logits
        lg, kv = lm.forward([tok], [L], [1], cache, L)
        for c, (k, v) in zip(cache, kv):
            c["K"][L] = k[0]
            c["V"][L] = v[0]
        L += 1
        logits = lg[0]

    for t in prompt:
        push(t)
    while len(out) < n_new:
        y, gap = smp.sample_row(logits, T, seed, 0, L)  # the token sampled here goes to position L
        gaps.append(gap)
        out.append(y)
        push(y)
    return out, cache, L, gaps


def sample_hybrid(lm: TinyLM, prompt: List[int], n_new: int, Lcap: int, cfg: dict, T: float, seed: int,
                  sharpen: float = 8.0, noise: float = 1.0):
    """Hybrid-tree decoding with sampling acceptance: the target's sample at every node, then the
    greedy rule on the samples.  Returns (tokens, cache, L, per-step records, perturbed-score gaps)."""
    rng = np.random.default_rng(seed + 7)
    cache = lm.new_cache(Lcap)
    L = 0
    for t in prompt[:-1]:
        _, kv = lm.forward([t], [L], [1], cache, L)
        for c, (k, v) in zip(cache, kv):
            c["K"][L] = k[0]
            c["V"][L] = v[0]
        L += 1
    root = prompt[-1]
    M_succ, M_cnt = um.empty_M(lm.V, cfg["W"])
    out: List[int] = []
    steps, gaps = [], []
    while len(out) < n_new:
        def row_fn(d, f, path, L=L):
            chain = [(1 << (i + 1)) - 1 for i in range(len(path))]
            lg, _ = lm.forward(path, [L + i for i in range(len(path))], chain, cache, L)
            return (sharpen * lg[-1] + rng.normal(0.0, noise, lm.V)).astype(np.float32)

        res = tr.draft_tree(row_fn, root, cfg)
        nodes = tr.retained_draft(res, cfg)
        ret = tr.retrieve(root, M_succ, cfg["tmpl_parent"], cfg["tmpl_rank"])
        tree = tr.merge(root, nodes, ret, cfg["tmpl_parent"], res.stage, L, cfg)
        logits, kv = lm.forward([max(t, 0) for t in tree.tok], tree.pos, tree.mask, cache, L)
        y, gap = smp.sample_tree(logits[None], np.array(tree.pos)[None], T, seed)
        g, n, path, out_tok, bonus = acc.accept_from_argmax(y[0], tree.tok, tree.parent, tree.depth)
        gaps.extend(gap[0][p] for p in path)
        for c, (k, v) in zip(cache, kv):
            for t, p in enumerate(path):
                c["K"][L + t] = k[p]
                c["V"][L + t] = v[p]
        L += n
        out.extend(out_tok)
        root = bonus
        M_succ, M_cnt = um.update_M(M_succ, M_cnt, np.array(tree.tok), np.array(g))
        steps.append(dict(stage=res.stage, acc_len=n,
                          retrieved_accepted=sum(1 for p in path if p >= tree.n_draft)))
    return out[:n_new], cache, L, steps, gaps

