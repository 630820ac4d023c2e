"""The attention kernels' failure path: a bounded wait that runs out.

Every wait of the tensor-core attention kernels on one of their pipeline
barriers is bounded.  When a bound runs out the CTA sets
GRAFT_STATUS_TIMEOUT, stops issuing work, waits (with fixed bounds) for the
loads and tensor-core products it already issued, frees its tensor memory
and exits, so the GPU stays usable.  GraftAttnTuning.wait_ns shortens the
pipeline bound to a few nanoseconds, so the first waits run out on small,
valid inputs (every load stays in bounds and completes; only the waiting is
cut short).  The test checks that the call returns with the TIMEOUT bit set
and that the next normal call on the same stream, with a re-zeroed
workspace, is correct: tensor memory was released and the context is fine.
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from tests.helpers import assert_attention_close, gb, to_np
from tree_verification_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(B, Hq, Hkv, Kmax, Ls, Lcap, seed):
    wl = synth.WORKLOADS["llama3_8b"].scaled(B=B, Hq=Hq, Hkv=Hkv, Kmax=Kmax, seed=seed, L=(0, 0))
    Q, Kc, Vc, Kt, Vt = synth.layer_tensors(wl, 0, DEV, Lcap=Lcap)
    masks = np.array([[(1 << (i + 1)) - 1 for i in range(Kmax)]] * B, dtype=np.uint64)  # chains
    return Q, Kc, Vc, Kt, Vt, torch.tensor(Ls, dtype=torch.int32), masks


@pytest.mark.parametrize("kernel,tuning,shape", [
    ("two-tile", dict(tiles=2, persist_ctas=-1), (1, 8, 2, 32, [512], 576)),
    ("one-tile, split keys", dict(tiles=1, persist_ctas=-1, min_chunk=256), (2, 32, 8, 64, [4096, 777], 4160)),
    ("persistent, stream schedule", dict(tiles=2, persist_ctas=3, min_chunk=1000000, split=1),
     (3, 32, 8, 64, [1500, 300, 129], 1536)),
    ("persistent, whole items", dict(tiles=2, persist_ctas=3, min_chunk=256),
     (3, 32, 8, 64, [4096, 0, 2300], 4160)),
])
def test_bounded_wait_runs_out_and_the_device_stays_usable(kernel, tuning, shape):
    B, Hq, Hkv, Kmax, Ls, Lcap = shape
    Q, Kc, Vc, Kt, Vt, L, masks = _case(B, Hq, Hkv, Kmax, Ls, Lcap, seed=B + Kmax)
    mask_d = torch.from_numpy(masks.view(np.int64)).to(DEV)
    ws = torch.zeros(max(1, gb().graft_tree_attention_workspace_size(B, Hq, Hkv, Kmax, Lcap, tuning)),
                     dtype=torch.uint8, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gb().graft_tree_attention(Q, Kc, Vc, Kt, Vt, L.to(DEV), mask_d, 1 / math.sqrt(128), status=status, ws=ws,
                              tuning=dict(tuning, wait_ns=2))
    torch.cuda.synchronize()
    assert int(status.item()) & gb().STATUS_TIMEOUT, f"{kernel}: no wait ran out"
    # the same stream again, normally: the workspace is zeroed anew (an aborted call may leave arrival
    # counters behind, as graft.h says)
    ws.zero_()
    status.zero_()
    O = gb().graft_tree_attention(Q, Kc, Vc, Kt, Vt, L.to(DEV), mask_d, 1 / math.sqrt(128), status=status, ws=ws,
                                  tuning=tuning)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oatt.tree_attention(to_np(Q), to_np(Kc), to_np(Vc), to_np(Kt), to_np(Vt), L.numpy(), masks,
                              1 / math.sqrt(128))
    assert_attention_close(to_np(O), ref)
