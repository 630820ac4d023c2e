"""VerifyStep with its inputs streamed in: the inputs_ready hook orders each stage after the copy
of that stage's inputs (drafter logits, then each layer's Q and tree K/V, then the target logits)
on another stream, and the step's results equal those of the same step on resident inputs."""
import numpy as np
import pytest
import torch

from tests.helpers import gb, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(wl, n_layers, synth):
    Lcap = wl.lcap()
    dl = synth.draft_logits(wl, DEV)
    roots, L0 = synth.root_tokens(wl).to(DEV), synth.prefix_lengths(wl).to(DEV)
    layers = [synth.layer_tensors(wl, l, DEV, Lcap=Lcap) for l in range(n_layers)]
    tl = synth.target_logits(wl, DEV)
    s_np, c_np = synth.zipf_M(wl.V, wl.W, wl.seed + 5)
    return Lcap, dl, roots, L0, layers, tl, s_np, c_np


def test_streamed_inputs_match_resident_inputs():
    from tree_verification_gb300 import synth
    from tree_verification_gb300.step import VerifyStep

    wl = synth.WORKLOADS["tiny"]
    n_layers = 3
    cfg = gb().graft_config_init(wl.Kmax, wl.D, wl.k, wl.V, wl.W, list(wl.checkpoints), wl.tau)
    Lcap, dl, roots, L0, layers, tl, s_np, c_np = _inputs(wl, n_layers, synth)

    def make_step():
        # each run compacts into its own copy of the caches
        return VerifyStep(cfg, wl.B, wl.Hq, wl.Hkv, n_layers, Lcap, DEV, [x[1].clone() for x in layers],
                          [x[2].clone() for x in layers], [x[3] for x in layers], [x[4] for x in layers])

    # resident inputs
    ref = make_step()
    Ms, Mc = torch.from_numpy(s_np).to(DEV), torch.from_numpy(c_np).to(DEV)
    L = L0.clone()
    ref.run(dl, roots, Ms, Mc, L, [x[0] for x in layers], tl)
    torch.cuda.synchronize()

    # streamed: device buffers start as garbage and are filled from pinned host copies on a copy stream
    host = {"dl": dl.cpu().pin_memory(), "roots": roots.cpu().pin_memory(), "L0": L0.cpu().pin_memory(),
            "tl": tl.cpu().pin_memory()}
    for l in range(n_layers):
        host[f"Q{l}"], host[f"Kt{l}"], host[f"Vt{l}"] = (layers[l][i].cpu().pin_memory() for i in (0, 3, 4))
    dev = {k: torch.full_like(v, 7, device=DEV) if v.dtype != torch.float32 else torch.full_like(v, float("nan"),
                                                                                                device=DEV)
           for k, v in host.items()}
    step = VerifyStep(cfg, wl.B, wl.Hq, wl.Hkv, n_layers, Lcap, DEV, [x[1].clone() for x in layers],
                      [x[2].clone() for x in layers], [dev[f"Kt{l}"] for l in range(n_layers)],
                      [dev[f"Vt{l}"] for l in range(n_layers)])
    stages = {"tree": ["dl", "roots", "L0"], "accept": ["tl"]}
    stages.update({l: [f"Q{l}", f"Kt{l}", f"Vt{l}"] for l in range(n_layers)})
    ready = {k: torch.cuda.Event() for k in stages}
    copy = torch.cuda.Stream()
    main = torch.cuda.current_stream()
    copy.wait_stream(main)
    with torch.cuda.stream(copy):
        for k, names in stages.items():
            for n in names:
                dev[n].copy_(host[n], non_blocking=True)
            ready[k].record()
    seen = []

    def inputs_ready(k):
        seen.append(k)
        main.wait_event(ready[k])
        if k == "tree":
            L.copy_(dev["L0"])

    Ms2, Mc2 = torch.from_numpy(s_np).to(DEV), torch.from_numpy(c_np).to(DEV)
    L = torch.empty_like(L0)
    step.run(dev["dl"], dev["roots"], Ms2, Mc2, L, [dev[f"Q{l}"] for l in range(n_layers)], dev["tl"],
             inputs_ready=inputs_ready)
    torch.cuda.synchronize()
    assert seen == ["tree"] + list(range(n_layers)) + ["accept"]
    assert int(step.status.item()) == 0 and int(ref.status.item()) == 0
    for k in ("tok", "parent", "depth", "pos", "mask"):
        assert torch.equal(step.tree[k], ref.tree[k]), k
    for k in ("acc_len", "out_tok", "bonus"):
        assert torch.equal(step.acc[k], ref.acc[k]), k
    assert torch.equal(step.O, ref.O)
    assert torch.equal(Ms2, Ms) and torch.equal(Mc2, Mc)
    for l in range(n_layers):
        assert torch.equal(step.Kc[l], ref.Kc[l]) and torch.equal(step.Vc[l], ref.Vc[l])
