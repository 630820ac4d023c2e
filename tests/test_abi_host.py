"""Host-side checks of libgraft.so (no GPU needed).

The library must load, export every entry point include/graft.h declares,
reject invalid arguments before touching the device, and produce the same
budget split and retrieval envelope as the oracle.
"""
import ctypes
import os
import re

import pytest

from oracle import config as oconfig
from tests.helpers import gb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^\s*(?:int|const char\*|size_t|uint64_t)\s+(graft_\w+)\s*\(", text, re.M))
    return sorted(names)


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert len(names) >= 12
    lib = ctypes.CDLL(gb().lib_path())
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version():
    b = gb()
    assert b.graft_status_string(0) == "ok"
    assert "workspace" in b.graft_status_string(-3)
    assert b.graft_version() >= 100


@pytest.mark.parametrize("Kmax,D,k,V,W", [(32, 6, 4, 32000, 8), (64, 8, 8, 128256, 16), (64, 8, 8, 151936, 32),
                                          (16, 4, 3, 4096, 4), (6, 3, 2, 8, 2), (1, 1, 1, 10, 1), (64, 8, 16, 1000, 32)])
def test_config_matches_oracle(Kmax, D, k, V, W):
    cfg = gb().graft_config_init(Kmax, D, k, V, W, [0, 1, 5], 0.3).as_dict()
    ref = oconfig.make_config(Kmax=Kmax, D=D, k=k, V=V, W=W)
    assert cfg["checkpoints"] == ref["checkpoints"]
    assert cfg["K_draft"] == ref["K_draft"]
    assert cfg["tmpl_parent"] == ref["tmpl_parent"] and cfg["tmpl_rank"] == ref["tmpl_rank"]
    assert cfg["n_tmpl"] == len(ref["tmpl_parent"])


@pytest.mark.parametrize("Kmax,D,k,V,W", [(32, 6, 4, 32000, 8), (64, 8, 8, 128256, 16), (6, 3, 2, 8, 2)])
def test_config_without_retrieval_matches_oracle(Kmax, D, k, V, W):
    b = gb()
    cfg = b.graft_config_no_retrieval(b.graft_config_init(Kmax, D, k, V, W, [0, 1, 5], 0.3)).as_dict()
    ref = oconfig.make_config(Kmax=Kmax, D=D, k=k, V=V, W=W, no_retrieval=True)
    assert cfg["K_draft"] == ref["K_draft"] == [Kmax] * len(ref["K_draft"])
    assert cfg["n_tmpl"] == 0 and ref["tmpl_parent"] == []
    assert b.graft_config_validate(b.graft_config_no_retrieval(b.graft_config_init(Kmax, D, k, V, W))) == 0


def test_tuning_fields_are_checked():
    lib = gb().lib()
    b = gb()
    sz = ctypes.c_size_t()
    for bad in (dict(tiles=3), dict(min_chunk=-1), dict(persist_ctas=-2), dict(reserved=(ctypes.c_int32 * 3)(0, 1)), dict(split=2), dict(split=-1), dict(wait_ns=-5)):
        t = b.GraftAttnTuning()
        for k, v in bad.items():
            setattr(t, k, v)
        assert lib.graft_tree_attention_workspace_size_ex(1, 8, 2, 128, 32, 512, ctypes.byref(t), ctypes.byref(sz)) == -1
    # no tuning (NULL) and an all-zero tuning plan the same workspace
    assert lib.graft_tree_attention_workspace_size_ex(2, 32, 8, 128, 64, 4160, None, ctypes.byref(sz)) == 0
    n0 = sz.value
    t = b.GraftAttnTuning()
    assert lib.graft_tree_attention_workspace_size_ex(2, 32, 8, 128, 64, 4160, ctypes.byref(t), ctypes.byref(sz)) == 0
    assert sz.value == n0


def test_config_rejects_bad():
    b = gb()
    with pytest.raises(b.GraftError):
        b.graft_config_init(65, 8, 8, 1000, 16)
    with pytest.raises(b.GraftError):
        b.graft_config_init(64, 2, 2, 1000, 16)  # dense draft smaller than Kmax - 1
    with pytest.raises(b.GraftError):
        b.graft_config_init(64, 8, 8, 1000, 33)
    cfg = b.graft_config_init(64, 8, 8, 1000, 16)
    cfg.K_draft[cfg.n_checkpoints] = 63
    assert b.graft_config_validate(cfg) == -1


def test_invalid_arguments_return_codes_without_launch():
    lib = gb().lib()
    sz = ctypes.c_size_t()
    assert lib.graft_tree_attention_workspace_size(1, 8, 2, 64, 32, 512, ctypes.byref(sz)) == -2  # head_dim
    assert lib.graft_tree_attention_workspace_size(1, 8, 3, 128, 32, 512, ctypes.byref(sz)) == -1  # Hq % Hkv
    assert lib.graft_tree_attention_workspace_size(1, 64, 4, 128, 65, 512, ctypes.byref(sz)) == -2  # Kmax
    assert lib.graft_tree_attention_workspace_size(1, 64, 1, 128, 64, 512, ctypes.byref(sz)) == -2  # rows
    # null pointers are refused before any launch
    assert lib.graft_tree_attention(1, 8, 2, 128, 32, None, None, None, 512, None, None, None, None,
                                    ctypes.c_float(1.0), None, None, None, 0, None) == -1
    assert lib.graft_update_M(None, None, 10, 4, None, None, 5, None, None, 0, None) == -1
    assert lib.graft_update_M(None, None, 10, 40, None, None, 5, None, None, 0, None) == -2
    # a zero-size batch is a no-op
    assert lib.graft_update_M(None, None, 10, 4, None, None, 0, None, None, 0, None) == 0
    assert lib.graft_accept_compact_workspace_size(4, 65, 100, ctypes.byref(sz)) == -2
    assert lib.graft_update_M_workspace_size(1000, ctypes.byref(sz)) == 0 and sz.value > 0


def test_workspace_checks():
    lib = gb().lib()
    b = gb()
    cfg = b.graft_config_init(32, 6, 4, 32000, 8)
    need = b.graft_build_tree_workspace_size(cfg, 2)
    assert need > 0
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: the call fails the size check first
    rc = lib.graft_build_tree(ctypes.byref(cfg), 2, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                              None, fake, need - 1, None)
    assert rc == -3
    rc = lib.graft_build_tree(ctypes.byref(cfg), 2, fake, fake, fake, fake, fake, fake, fake, fake, fake, fake,
                              None, ctypes.c_void_p(0x1010), need, None)  # misaligned workspace
    assert rc == -3
