"""Per-call timing of graft_tree_attention on one synthetic workload.

    python -m tree_verification_gb300.attn_bench WORKLOAD [--layers N] [--reps R] [--lcap C]

Builds N layers of the workload's synthetic Q / KV cache / tree KV (distinct
buffers per layer, so repeated calls are not served from L2), captures the N
layer calls in one CUDA graph, replays it R times after a warm-up and prints
one line: microseconds per call, the call's compulsory bytes (prefix and tree
K/V, Q in, O out) over that time, and the device status word.  The tree mask
is a chain (every node sees its ancestors), which does not change the work.
--lcap sizes the KV cache for C positions instead of the workload's prefix
plus its decode steps (the prefixes stay the same), to show that the time
follows the prefix lengths rather than the cache capacity.
"""
from __future__ import annotations

import argparse
import math

import numpy as np
import torch

from . import binding as gb
from . import synth


def time_calls(wl, n_layers: int, reps: int, Lcap: int = 0, dev=None):
    """Microseconds per graft_tree_attention call of workload wl (n_layers distinct layers captured
    in one CUDA graph, replayed reps times after a warm-up), the call's compulsory bytes and the
    device status word."""
    dev = torch.device("cuda") if dev is None else dev
    Lcap = max(Lcap, wl.lcap()) if Lcap else wl.lcap()
    L = synth.prefix_lengths(wl).to(dev)
    layers = [synth.layer_tensors(wl, l, dev, Lcap=Lcap) for l in range(n_layers)]
    chain = np.array([[(1 << (i + 1)) - 1 for i in range(wl.Kmax)]] * wl.B, dtype=np.uint64)
    mask = torch.from_numpy(chain.view(np.int64)).to(dev)
    ws = torch.empty(max(1, gb.graft_tree_attention_workspace_size(wl.B, wl.Hq, wl.Hkv, wl.Kmax, Lcap)),
                     dtype=torch.uint8, device=dev)
    O = torch.empty_like(layers[0][0])
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    scale = 1.0 / math.sqrt(gb.HEAD_DIM)

    def run():
        for (Q, Kc, Vc, Kt, Vt) in layers:
            gb.graft_tree_attention(Q, Kc, Vc, Kt, Vt, L, mask, scale, O=O, ws=ws, status=status)

    run()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(reps):
        graph.replay()
    stop.record()
    stop.synchronize()
    us = start.elapsed_time(stop) * 1000.0 / (reps * n_layers)
    d = gb.HEAD_DIM
    nbytes = (2 * int(L.sum()) * wl.Hkv * d * 2 + 2 * wl.B * wl.Kmax * wl.Hkv * d * 2
              + 2 * wl.B * wl.Kmax * wl.Hq * d * 2)
    st = int(status.item())
    del layers, ws, O
    return us, nbytes, st


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("workload", choices=sorted(synth.WORKLOADS))
    p.add_argument("--layers", type=int, default=4)
    p.add_argument("--reps", type=int, default=20)
    p.add_argument("--lcap", type=int, default=0)
    args = p.parse_args(argv)
    wl = synth.WORKLOADS[args.workload]
    us, nbytes, st = time_calls(wl, args.layers, args.reps, args.lcap)
    print(f"{args.workload}: {us:.2f} us per call, {nbytes / 1e6:.2f} MB per call, "
          f"{nbytes / us / 1e3:.0f} GB/s, status {st}")


if __name__ == "__main__":
    main()
