"""One hybrid-tree verify step through the C ABI, with preallocated buffers.

``VerifyStep`` owns the outputs and workspaces of the four library calls
and runs them in the Graft article's order on one CUDA stream:

    graft_build_tree  ->  graft_tree_attention x n_layers  ->
    graft_accept_compact  ->  M update

With ``temperature`` > 0 the step verifies by sampling: graft_sample_tokens
draws the target's sample at every node (keyed by ``seed`` and position)
and graft_accept_compact accepts on those samples; otherwise it is greedy.

The M update follows ``m_policy``: "tree" adds every tree node's (token,
target argmax) pair (graft_update_M); "emitted" adds the bigrams of the
tokens the step emitted (graft_update_M_emitted), the prompt-evidence policy
that ``prefill_M`` seeds with the prompt's bigrams; "both" does both.

Because every buffer is fixed, a whole step can be captured once in a CUDA
graph and replayed, which removes the per-layer host launch cost.  The
caller owns the model-side tensors: drafter and target logits, per-layer
Q / tree KV / KV caches, the cache lengths and the table M.
"""
from __future__ import annotations

import math
from typing import Callable, List, Optional, Sequence

import torch

from . import binding as gb


class VerifyStep:
    def __init__(self, cfg: gb.GraftConfig, B: int, Hq: int, Hkv: int, n_layers: int, Lcap: int, device,
                 Kc: Sequence[torch.Tensor], Vc: Sequence[torch.Tensor], Kt: Sequence[torch.Tensor],
                 Vt: Sequence[torch.Tensor], m_policy: str = "tree", temperature: float = 0.0, seed: int = 0):
        if m_policy not in ("tree", "emitted", "both"):
            raise ValueError("m_policy must be 'tree', 'emitted' or 'both'")
        self.m_policy = m_policy
        self.temperature, self.seed = float(temperature), int(seed)
        self.cfg, self.B, self.Hq, self.Hkv, self.n_layers, self.Lcap = cfg, B, Hq, Hkv, n_layers, Lcap
        self.device = torch.device(device)
        K, dev = cfg.Kmax, self.device
        i32 = dict(dtype=torch.int32, device=dev)
        self.tree = dict(tok=torch.empty(B, K, **i32), parent=torch.empty(B, K, **i32),
                         depth=torch.empty(B, K, **i32), pos=torch.empty(B, K, **i32),
                         mask=torch.empty(B, K, dtype=torch.int64, device=dev), stage=torch.empty(B, **i32))
        self.acc = dict(argmax=torch.empty(B, K, **i32), acc_len=torch.empty(B, **i32),
                        path=torch.empty(B, K, **i32), out_tok=torch.empty(B, K, **i32),
                        bonus=torch.empty(B, **i32))
        self.status = torch.zeros(1, **i32)
        u8 = dict(dtype=torch.uint8, device=dev)
        # zero-filled once: the tree build's grid barrier and the attention workspace's arrival
        # counters must start at zero (every call leaves them at zero)
        self.ws_tree = torch.zeros(max(1, gb.graft_build_tree_workspace_size(cfg, B)), **u8)
        self.ws_attn = torch.zeros(max(1, gb.graft_tree_attention_workspace_size(B, Hq, Hkv, K, Lcap)), **u8)
        self.ws_acc = torch.empty(max(1, gb.graft_accept_compact_workspace_size(B, K, cfg.V)), **u8)
        self.ws_upd = torch.empty(max(1, gb.graft_update_M_workspace_size(B * K)), **u8)
        self.ws_emit = torch.empty(max(1, gb.graft_update_M_emitted_workspace_size(B, K)), **u8)
        self.ws_smp = torch.empty(max(1, gb.graft_sample_tokens_workspace_size(B, K, cfg.V)), **u8)
        self.O = torch.empty(B, K, Hq, gb.HEAD_DIM, dtype=torch.bfloat16, device=dev)
        self.Kc, self.Vc, self.Kt, self.Vt = list(Kc), list(Vc), list(Kt), list(Vt)
        self.Kc_ptrs = gb.layer_pointers(self.Kc, dev)
        self.Vc_ptrs = gb.layer_pointers(self.Vc, dev)
        self.Kt_ptrs = gb.layer_pointers(self.Kt, dev)
        self.Vt_ptrs = gb.layer_pointers(self.Vt, dev)
        self.scale = 1.0 / math.sqrt(gb.HEAD_DIM)
        self.graph: Optional[torch.cuda.CUDAGraph] = None

    def run(self, draft_logits, root_tok, M_succ, M_cnt, L, Q: Sequence[torch.Tensor], target_logits,
            attn_layers: Optional[Sequence[int]] = None,
            inputs_ready: Optional[Callable[[object], None]] = None) -> None:
        """Enqueue one step on the current stream (asynchronous).

        ``inputs_ready``, if given, is called just before each stage is enqueued, with "tree"
        (drafter logits, root tokens, lengths), then each layer index (that layer's Q and tree
        K/V), then "accept" (target logits), so the caller can order the stream after whatever
        produces that stage's inputs (for example a copy on another stream) instead of waiting
        for all of them before the step starts.
        """
        if inputs_ready is not None:
            inputs_ready("tree")
        gb.graft_build_tree(self.cfg, draft_logits, root_tok, M_succ, L, out=self.tree, status=self.status,
                            ws=self.ws_tree)
        for l in (range(self.n_layers) if attn_layers is None else attn_layers):
            if inputs_ready is not None:
                inputs_ready(l)
            gb.graft_tree_attention(Q[l], self.Kc[l], self.Vc[l], self.Kt[l], self.Vt[l], L, self.tree["mask"],
                                    self.scale, O=self.O, status=self.status, ws=self.ws_attn)
        if inputs_ready is not None:
            inputs_ready("accept")
        if self.temperature > 0.0:
            gb.graft_sample_tokens(target_logits, self.tree["pos"], self.temperature, self.seed,
                                   sampled=self.acc["argmax"], ws=self.ws_smp)
            gb.graft_accept_compact(None, self.tree["tok"], self.tree["parent"], self.tree["depth"],
                                    self.Kc_ptrs, self.Vc_ptrs, self.Kt_ptrs, self.Vt_ptrs, self.n_layers, self.Hkv,
                                    self.Lcap, L, out=self.acc, status=self.status, ws=self.ws_acc,
                                    argmax=self.acc["argmax"], V=self.cfg.V)
        else:
            gb.graft_accept_compact(target_logits, self.tree["tok"], self.tree["parent"], self.tree["depth"],
                                    self.Kc_ptrs, self.Vc_ptrs, self.Kt_ptrs, self.Vt_ptrs, self.n_layers, self.Hkv,
                                    self.Lcap, L, out=self.acc, status=self.status, ws=self.ws_acc)
        if self.m_policy in ("tree", "both"):
            gb.graft_update_M(M_succ, M_cnt, self.tree["tok"].view(-1), self.acc["argmax"].view(-1),
                              status=self.status, ws=self.ws_upd)
        if self.m_policy in ("emitted", "both"):
            gb.graft_update_M_emitted(M_succ, M_cnt, self.tree["tok"], self.acc["out_tok"], self.acc["acc_len"],
                                      status=self.status, ws=self.ws_emit)

    def prefill_M(self, M_succ, M_cnt, prompt_tokens) -> None:
        """Seed M with the prompt's bigrams (the prompt-evidence policy's starting table)."""
        gb.graft_seed_M_from_tokens(M_succ, M_cnt, prompt_tokens, status=self.status)

    def capture(self, *args, **kw) -> torch.cuda.CUDAGraph:
        """Capture run(*args) into a CUDA graph (the arguments' storage is baked in)."""
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.run(*args, **kw)  # warm the launch path once outside capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize(self.device)
        with torch.cuda.graph(g):
            self.run(*args, **kw)
        self.graph = g
        return g
