"""graft_update_M_noalloc against graft_update_M on the GPU.

The no-allocation entry point serves callers that cannot hand the library a
workspace (a plug-in that only receives tensors from its host framework, or
a serving loop that must avoid cudaMalloc's device-wide synchronisation).
It keeps its scratch in a fixed device array of the library, so this test
checks that two calls in a row — the second one reading a scratch array the
first one left dirty — give exactly what the workspace entry point gives,
and that batches above the array's limit are refused.  The file name sorts
last so that a run stopping at the first failure has run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests.helpers import gb

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _table(V, W, rng, fill):
    succ = np.full((V, W), -1, np.int32)
    cnt = np.zeros((V, W), np.int32)
    for t in range(V):
        k = int(rng.integers(0, fill + 1))
        toks = rng.choice(V, k, replace=False)
        cs = rng.integers(1, 6, k)
        order = sorted(range(k), key=lambda j: (-cs[j], toks[j]))
        succ[t, :k] = toks[order]
        cnt[t, :k] = cs[order]
    return succ, cnt


def test_two_calls_match_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.fail("GPU test needs a CUDA device")
    b = gb()
    rng = np.random.default_rng(123)
    V, W = 3000, 16
    succ, cnt = _table(V, W, rng, 12)
    ref_s, ref_c = torch.from_numpy(succ).to(DEV), torch.from_numpy(cnt).to(DEV)
    got_s, got_c = ref_s.clone(), ref_c.clone()
    status = torch.zeros(2, dtype=torch.int32, device=DEV)
    for n in (b.NOALLOC_MAX_PAIRS, 777):  # a full batch, then a smaller one over the dirty scratch
        src = torch.from_numpy(rng.integers(0, V, n).astype(np.int32)).to(DEV)
        dst = torch.from_numpy(rng.integers(0, V // 3, n).astype(np.int32)).to(DEV)
        b.graft_update_M(ref_s, ref_c, src, dst, status=status[0:1])
        b.graft_update_M_noalloc(got_s, got_c, src, dst, status=status[1:2])
        torch.cuda.synchronize()
        assert status.tolist() == [0, 0]
        assert torch.equal(got_s, ref_s) and torch.equal(got_c, ref_c)


def test_oversized_batch_is_refused_through_the_c_abi():
    b = gb()
    lib = b.lib()
    s = torch.zeros(10, 4, dtype=torch.int32, device=DEV)
    c = torch.zeros(10, 4, dtype=torch.int32, device=DEV)
    pairs = torch.zeros(b.NOALLOC_MAX_PAIRS + 1, dtype=torch.int32, device=DEV)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.graft_update_M_noalloc(p(s), p(c), 10, 4, p(pairs), p(pairs), pairs.numel(), None, None)
    assert rc == -2  # GRAFT_ERR_UNSUPPORTED_SHAPE
    torch.cuda.synchronize()
    assert int(s.abs().sum()) == 0 and int(c.abs().sum()) == 0
