"""One whole hybrid-tree verify step on the CPU (oracle, test infrastructure).

Composes the stages in the order the Graft article's method paragraph gives
them: prune the draft, fill the retrieval template from M, merge into one
Kmax-node tree, verify it with tree attention in one target forward (one
call per layer), accept the longest greedy path and compact its KV, then
update M from the verified tree.
"""
from __future__ import annotations

from typing import List, Optional, Sequence

import numpy as np

from . import accept as acc
from . import attention as att
from . import tree as tr
from . import update_m as um


def verify_step(cfg: dict, draft_logits, root_tok, M_succ, M_cnt, L, Q_layers: Sequence,
                Kc_layers: List, Vc_layers: List, Kt_layers: Sequence, Vt_layers: Sequence,
                target_logits, scale: float, attn_layers: Optional[Sequence[int]] = None) -> dict:
    """Run one step.  Caches are updated in place; returns every output.

    ``attn_layers`` restricts the attention (whose outputs feed nothing else
    in a synthetic step) to a subset of layers; compaction always covers all.
    """
    tree = tr.build_tree_batch(draft_logits, root_tok, M_succ, L, cfg)
    outs = {}
    layers = range(len(Q_layers)) if attn_layers is None else attn_layers
    for l in layers:
        outs[l] = att.tree_attention(Q_layers[l], Kc_layers[l], Vc_layers[l], Kt_layers[l],
                                     Vt_layers[l], L, tree["mask"], scale)
    a = acc.accept_batch(target_logits, tree)
    L_new = None
    for l in range(len(Kc_layers)):
        L_new = acc.compact(Kc_layers[l], Vc_layers[l], Kt_layers[l], Vt_layers[l],
                            np.asarray(L, np.int64), a["path"], a["acc_len"])
    succ, cnt = um.update_M(M_succ, M_cnt, tree["tok"].reshape(-1), a["argmax"].reshape(-1))
    return dict(tree=tree, attn=outs, accept=a, L=L_new, M_succ=succ, M_cnt=cnt)
