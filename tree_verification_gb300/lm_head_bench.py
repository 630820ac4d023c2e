"""Timing of the fused lm_head argmax and sampling kernels on synthetic inputs.

    python -m tree_verification_gb300.lm_head_bench N D_MODEL V [--reps R]

H [N][D_MODEL] and W [V][D_MODEL] are bf16 N(0,1).  Prints microseconds per
call for graft_lm_head_argmax and graft_lm_head_sample with the achieved
tensor throughput (2 N D_MODEL V flops) and operand bandwidth (H and W bf16).
"""
from __future__ import annotations

import argparse

import torch

from . import binding as gb


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("N", type=int)
    p.add_argument("d_model", type=int)
    p.add_argument("V", type=int)
    p.add_argument("--reps", type=int, default=10)
    a = p.parse_args(argv)
    g = torch.Generator(device="cuda").manual_seed(0)
    H = torch.randn(a.N, a.d_model, device="cuda", generator=g).to(torch.bfloat16)
    W = torch.randn(a.V, a.d_model, device="cuda", generator=g).to(torch.bfloat16)
    out = torch.empty(a.N, dtype=torch.int32, device="cuda")
    mx = torch.empty(a.N, dtype=torch.float32, device="cuda")
    pos = torch.arange(a.N, dtype=torch.int32, device="cuda").view(1, a.N)
    ws = torch.empty(max(1, gb.graft_lm_head_argmax_workspace_size(a.N)), dtype=torch.uint8, device="cuda")
    calls = {"argmax": lambda: gb.graft_lm_head_argmax(H, W, out, mx, None, ws),
             "sample": lambda: gb.graft_lm_head_sample(H, W, pos, 1.0, 7, sampled=out, ws=ws)}
    flops = 2.0 * a.N * a.d_model * a.V
    nbytes = (H.numel() + W.numel()) * 2
    for name, fn in calls.items():
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(a.reps):
            fn()
        e.record()
        e.synchronize()
        us = s.elapsed_time(e) * 1000.0 / a.reps
        print(f"{name} N={a.N} d={a.d_model} V={a.V}: {us:.1f} us, {flops / us / 1e6:.0f} TFLOP/s, "
              f"{nbytes / us / 1e3:.0f} GB/s")


if __name__ == "__main__":
    main()
