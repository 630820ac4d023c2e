"""Helpers shared by the tests: library build, oracle config views, tolerance checks."""
import functools

import numpy as np
import torch

from oracle import config as oconfig

# Attention tolerance: elementwise |gpu - ref| <= 1e-2 and, per tensor,
# max|gpu - ref| / max|ref| <= 2e-2 (bf16 inputs, fp32 accumulation, fp64 reference).
ATOL = 1e-2
RTOL_MAX = 2e-2
# Float-decided integer outputs are compared bit-exactly only when every
# decision clears this margin (float32 score error is far below it).
MARGIN = 5e-5


@functools.lru_cache(maxsize=1)
def built_lib():
    from tree_verification_gb300 import _build
    return _build.build()


def gb():
    built_lib()
    from tree_verification_gb300 import binding
    return binding


def oracle_cfg(wl, tau=None, checkpoints=None, no_retrieval=False):
    return oconfig.make_config(Kmax=wl.Kmax, D=wl.D, k=wl.k, V=wl.V, W=wl.W,
                               checkpoints=wl.checkpoints if checkpoints is None else checkpoints,
                               tau=wl.tau if tau is None else tau, no_retrieval=no_retrieval)


def lib_cfg(wl, tau=None, checkpoints=None):
    cps = [d for d in (wl.checkpoints if checkpoints is None else checkpoints)]
    return gb().graft_config_init(wl.Kmax, wl.D, wl.k, wl.V, wl.W, cps, wl.tau if tau is None else tau)


def assert_attention_close(gpu: np.ndarray, ref: np.ndarray):
    err = np.abs(gpu.astype(np.float64) - ref)
    assert err.max() <= ATOL, f"max abs error {err.max():.3e}"
    rel = err.max() / max(np.abs(ref).max(), 1e-30)
    assert rel <= RTOL_MAX, f"max error / max |ref| = {rel:.3e}"
    return float(err.max()), float(rel)


def to_np(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()


def mask_to_u64(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint64)


_WARM = {}


def warm_M(wl):
    """The oracle's table after the long-context warm-up: five multiset updates, each with every adjacent
    pair of the workload's seeded 65536-token stream.  Cached per workload name."""
    from oracle import update_m as oupd
    from tree_verification_gb300 import synth
    if wl.name not in _WARM:
        src, dst = synth.stream_pairs(synth.token_stream(wl.Lmax, wl.V, wl.seed + 41))
        s, c = synth.empty_M(wl.V, wl.W)
        for _ in range(5):
            s, c = oupd.update_M(s, c, src, dst)
        _WARM[wl.name] = (s, c)
    return _WARM[wl.name]


def initial_M(wl):
    """A workload's starting table as host arrays: Zipf counts, the warm-up table, or empty."""
    from tree_verification_gb300 import synth
    if wl.M_init == "zipf":
        return synth.zipf_M(wl.V, wl.W, wl.seed + 5)
    if wl.M_init == "warm":
        s, c = warm_M(wl)
        return s.copy(), c.copy()
    return synth.empty_M(wl.V, wl.W)
