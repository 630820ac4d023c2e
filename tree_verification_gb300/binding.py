"""Thin Python binding of libgraft.so (argument marshalling only).

Every function here has the name of the C entry point it wraps and does no
arithmetic of its own: it checks dtypes, devices and contiguity, allocates
outputs and workspaces with PyTorch on the input's device, and passes raw
device pointers plus the current CUDA stream.  Every step of the verify
path runs in the library's kernels; there is no CPU fallback, and importing
a function whose library is missing raises immediately.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libgraft.so")

GRAFT_OK = 0
ERR_CUDA = -4
STATUS_TOKEN_RANGE = 1
STATUS_CACHE_OVERFLOW = 2
STATUS_LENGTH = 4
STATUS_TREE = 8
STATUS_TIMEOUT = 16
STATUS_WORKSPACE = 32
EMPTY_TOKEN = -1

MAX_KMAX = 64
MAX_CHECKPOINTS = 4
HEAD_DIM = 128


class GraftConfig(ctypes.Structure):
    """Mirror of the C struct GraftConfig (graft.h)."""
    _fields_ = [
        ("Kmax", ctypes.c_int32), ("D", ctypes.c_int32), ("k", ctypes.c_int32),
        ("V", ctypes.c_int32), ("W", ctypes.c_int32),
        ("n_checkpoints", ctypes.c_int32),
        ("checkpoint", ctypes.c_int32 * MAX_CHECKPOINTS),
        ("tau", ctypes.c_float * MAX_CHECKPOINTS),
        ("K_draft", ctypes.c_int32 * (MAX_CHECKPOINTS + 1)),
        ("n_tmpl", ctypes.c_int32),
        ("tmpl_parent", ctypes.c_int32 * MAX_KMAX),
        ("tmpl_rank", ctypes.c_int32 * MAX_KMAX),
    ]

    def as_dict(self) -> dict:
        n = self.n_checkpoints
        return dict(Kmax=self.Kmax, D=self.D, k=self.k, V=self.V, W=self.W,
                    checkpoints=list(self.checkpoint[:n]), tau=list(self.tau[:n]),
                    K_draft=list(self.K_draft[: n + 1]), n_tmpl=self.n_tmpl,
                    tmpl_parent=list(self.tmpl_parent[: self.n_tmpl]),
                    tmpl_rank=list(self.tmpl_rank[: self.n_tmpl]))


class GraftAttnTuning(ctypes.Structure):
    """Mirror of the C struct GraftAttnTuning (graft.h): explicit launch-plan overrides of the tree
    attention (0 in a field keeps the default plan)."""
    _fields_ = [("tiles", ctypes.c_int32), ("min_chunk", ctypes.c_int32), ("persist_ctas", ctypes.c_int32),
                ("split", ctypes.c_int32), ("wait_ns", ctypes.c_int32), ("reserved", ctypes.c_int32 * 3)]


class GraftError(RuntimeError):
    pass


_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_SIGNATURES = {
    "graft_config_init": [ctypes.POINTER(GraftConfig), _I, _I, _I, _I, _I, _I, _P, _P],
    "graft_config_validate": [ctypes.POINTER(GraftConfig)],
    "graft_config_no_retrieval": [ctypes.POINTER(GraftConfig)],
    "graft_build_tree_workspace_size": [ctypes.POINTER(GraftConfig), _I, ctypes.POINTER(_SZ)],
    "graft_build_tree": [ctypes.POINTER(GraftConfig), _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "graft_build_tree_block": [ctypes.POINTER(GraftConfig), _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                               _P],
    "graft_retrieve": [ctypes.POINTER(GraftConfig), _I, _P, _P, _P, _P, _P],
    "graft_tree_attention_workspace_size": [_I, _I, _I, _I, _I, _I64, ctypes.POINTER(_SZ)],
    "graft_tree_attention": [_I, _I, _I, _I, _I, _P, _P, _P, _I64, _P, _P, _P, _P, ctypes.c_float, _P, _P, _P,
                             _SZ, _P],
    "graft_tree_attention_workspace_size_ex": [_I, _I, _I, _I, _I, _I64, ctypes.POINTER(GraftAttnTuning),
                                               ctypes.POINTER(_SZ)],
    "graft_tree_attention_ex": [_I, _I, _I, _I, _I, _P, _P, _P, _I64, _P, _P, _P, _P, ctypes.c_float, _P, _P,
                                ctypes.POINTER(GraftAttnTuning), _P, _SZ, _P],
    "graft_accept_compact_workspace_size": [_I, _I, _I, ctypes.POINTER(_SZ)],
    "graft_accept_compact": [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I64, _P, _P, _P, _P, _P, _P,
                             _P, _P, _SZ, _P],
    "graft_lm_head_argmax_workspace_size": [_I, ctypes.POINTER(_SZ)],
    "graft_lm_head_sample": [_I, _I, _I, _P, _P, _I, _P, ctypes.c_float, ctypes.c_uint64, _P, _P, _P, _SZ, _P],
    "graft_sample_tokens_workspace_size": [_I, _I, _I, ctypes.POINTER(_SZ)],
    "graft_sample_tokens": [_I, _I, _I, _P, _P, ctypes.c_float, ctypes.c_uint64, _P, _P, _SZ, _P],
    "graft_lm_head_argmax": [_I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "graft_update_M_workspace_size": [_I64, ctypes.POINTER(_SZ)],
    "graft_update_M": [_P, _P, _I, _I, _P, _P, _I64, _P, _P, _SZ, _P],
    "graft_update_M_noalloc": [_P, _P, _I, _I, _P, _P, _I64, _P, _P],
    "graft_update_M_emitted_workspace_size": [_I, _I, ctypes.POINTER(_SZ)],
    "graft_update_M_emitted": [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P],
    "graft_status_string": [_I],
    "graft_version": [],
    "graft_launch_count": [],
    "graft_last_cuda_error": [],
}


def lib_path() -> str:
    return _LIB_PATH


def lib():
    """Load libgraft.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise GraftError(f"{_LIB_PATH} is missing: build it with tree_verification_gb300._build.build()")
        L = ctypes.CDLL(_LIB_PATH)
        for name, args in _SIGNATURES.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = {"graft_status_string": ctypes.c_char_p, "graft_last_cuda_error": ctypes.c_char_p,
                          "graft_launch_count": ctypes.c_uint64}.get(name, ctypes.c_int)
        _lib = L
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != GRAFT_OK:
        msg = f"{what}: {lib().graft_status_string(rc).decode()} ({rc})"
        if rc == ERR_CUDA:
            msg += f" [{lib().graft_last_cuda_error().decode()}]"
        raise GraftError(msg)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _ws(nbytes: int, device, ws: Optional[torch.Tensor], zero: bool = False):
    if nbytes == 0:
        return None, 0
    if ws is None:
        ws = (torch.zeros if zero else torch.empty)(nbytes, dtype=torch.uint8, device=device)
    if ws.numel() < nbytes:
        raise ValueError("workspace too small")
    return ws, ws.numel()


def graft_config_init(Kmax: int, D: int, k: int, V: int, W: int, checkpoints: Sequence[int] = (0, 1, 5),
                      tau=0.3) -> GraftConfig:
    cps = list(checkpoints)
    taus = [float(tau)] * len(cps) if isinstance(tau, (int, float)) else [float(t) for t in tau]
    if len(taus) != len(cps):
        raise ValueError("one tau per checkpoint")
    cfg = GraftConfig()
    ca = (ctypes.c_int32 * max(1, len(cps)))(*cps)
    ta = (ctypes.c_float * max(1, len(taus)))(*taus)
    _check(lib().graft_config_init(ctypes.byref(cfg), Kmax, D, k, V, W, len(cps),
                                   ctypes.cast(ca, _P), ctypes.cast(ta, _P)), "graft_config_init")
    return cfg


def graft_config_no_retrieval(cfg: GraftConfig) -> GraftConfig:
    """The "w/o retrieval" ablation of cfg (K_ret = 0 at every stage), edited in place and returned."""
    _check(lib().graft_config_no_retrieval(ctypes.byref(cfg)), "graft_config_no_retrieval")
    return cfg


def graft_config_validate(cfg: GraftConfig) -> int:
    return lib().graft_config_validate(ctypes.byref(cfg))


def graft_build_tree_workspace_size(cfg: GraftConfig, B: int) -> int:
    n = _SZ()
    _check(lib().graft_build_tree_workspace_size(ctypes.byref(cfg), B, ctypes.byref(n)), "workspace size")
    return n.value


def graft_build_tree(cfg: GraftConfig, draft_logits, root_tok, M_succ, L, out: Optional[dict] = None,
                     status=None, ws=None, stream=None, block: bool = False) -> dict:
    """Drafter logits [B][D][k][V]; with block=True, block-drafter logits [B][D][V] (graft_build_tree_block)."""
    B = root_tok.shape[0]
    _need(draft_logits, "draft_logits", torch.float32, (B, cfg.D, cfg.V) if block else (B, cfg.D, cfg.k, cfg.V))
    _need(root_tok, "root_tok", torch.int32, (B,))
    _need(M_succ, "M_succ", torch.int32, (cfg.V, cfg.W))
    _need(L, "L", torch.int32, (B,))
    dev = root_tok.device
    if out is None:
        K = cfg.Kmax
        out = dict(tok=torch.empty(B, K, dtype=torch.int32, device=dev),
                   parent=torch.empty(B, K, dtype=torch.int32, device=dev),
                   depth=torch.empty(B, K, dtype=torch.int32, device=dev),
                   pos=torch.empty(B, K, dtype=torch.int32, device=dev),
                   mask=torch.empty(B, K, dtype=torch.int64, device=dev),
                   stage=torch.empty(B, dtype=torch.int32, device=dev))
    ws, nws = _ws(graft_build_tree_workspace_size(cfg, B), dev, ws, zero=True)
    fn = lib().graft_build_tree_block if block else lib().graft_build_tree
    _check(fn(ctypes.byref(cfg), B, _ptr(draft_logits), _ptr(root_tok), _ptr(M_succ), _ptr(L),
              _ptr(out["tok"]), _ptr(out["parent"]), _ptr(out["depth"]), _ptr(out["pos"]),
              _ptr(out["mask"]), _ptr(out["stage"]), _ptr(status), _ptr(ws), nws,
              _stream(stream)), "graft_build_tree")
    return out


def graft_retrieve(cfg: GraftConfig, root_tok, M_succ, ret_tok=None, status=None, stream=None):
    B = root_tok.shape[0]
    _need(root_tok, "root_tok", torch.int32, (B,))
    _need(M_succ, "M_succ", torch.int32, (cfg.V, cfg.W))
    if ret_tok is None:
        ret_tok = torch.empty(B, cfg.n_tmpl, dtype=torch.int32, device=root_tok.device)
    _check(lib().graft_retrieve(ctypes.byref(cfg), B, _ptr(root_tok), _ptr(M_succ), _ptr(ret_tok), _ptr(status),
                                _stream(stream)), "graft_retrieve")
    return ret_tok


def _tuning(tuning) -> Optional["GraftAttnTuning"]:
    if tuning is None or isinstance(tuning, GraftAttnTuning):
        return tuning
    t = GraftAttnTuning()
    for k, v in dict(tuning).items():
        setattr(t, k, int(v))
    return t


def graft_tree_attention_workspace_size(B: int, Hq: int, Hkv: int, Kmax: int, Lcap: int, tuning=None) -> int:
    """Workspace bytes of graft_tree_attention; ``tuning`` (a GraftAttnTuning or a dict of its fields)
    selects graft_tree_attention_workspace_size_ex."""
    n = _SZ()
    t = _tuning(tuning)
    if t is None:
        rc = lib().graft_tree_attention_workspace_size(B, Hq, Hkv, HEAD_DIM, Kmax, Lcap, ctypes.byref(n))
    else:
        rc = lib().graft_tree_attention_workspace_size_ex(B, Hq, Hkv, HEAD_DIM, Kmax, Lcap, ctypes.byref(t),
                                                          ctypes.byref(n))
    _check(rc, "workspace size")
    return n.value


def graft_tree_attention(Q, Kc, Vc, Kt, Vt, L, tree_mask, scale: float, O=None, status=None, ws=None,
                         stream=None, tuning=None):
    """Tree attention of one layer; ``tuning`` (a GraftAttnTuning or a dict of its fields) selects
    graft_tree_attention_ex with that launch plan."""
    B, Kmax, Hq, d = Q.shape
    Lcap, Hkv = Kc.shape[1], Kc.shape[2]
    _need(Q, "Q", torch.bfloat16)
    _need(Kc, "Kc", torch.bfloat16, (B, Lcap, Hkv, d))
    _need(Vc, "Vc", torch.bfloat16, (B, Lcap, Hkv, d))
    _need(Kt, "Kt", torch.bfloat16, (B, Kmax, Hkv, d))
    _need(Vt, "Vt", torch.bfloat16, (B, Kmax, Hkv, d))
    _need(L, "L", torch.int32, (B,))
    _need(tree_mask, "tree_mask", torch.int64, (B, Kmax))
    if O is None:
        O = torch.empty_like(Q)
    _need(O, "O", torch.bfloat16, Q.shape)
    t = _tuning(tuning)
    # the attention workspace starts zero-filled (its arrival counters); calls leave it that way
    ws, nws = _ws(graft_tree_attention_workspace_size(B, Hq, Hkv, Kmax, Lcap, t), Q.device, ws, zero=True)
    args = (B, Hq, Hkv, d, Kmax, _ptr(Q), _ptr(Kc), _ptr(Vc), Lcap, _ptr(Kt), _ptr(Vt), _ptr(L), _ptr(tree_mask),
            float(scale), _ptr(O), _ptr(status))
    if t is None:
        rc = lib().graft_tree_attention(*args, _ptr(ws), nws, _stream(stream))
    else:
        rc = lib().graft_tree_attention_ex(*args, ctypes.byref(t), _ptr(ws), nws, _stream(stream))
    _check(rc, "graft_tree_attention")
    return O


def graft_accept_compact_workspace_size(B: int, Kmax: int, V: int) -> int:
    n = _SZ()
    _check(lib().graft_accept_compact_workspace_size(B, Kmax, V, ctypes.byref(n)), "workspace size")
    return n.value


def layer_pointers(tensors: Sequence[torch.Tensor], device) -> torch.Tensor:
    """A device int64 array of the tensors' data pointers (the layer tables of graft_accept_compact)."""
    return torch.tensor([t.data_ptr() for t in tensors], dtype=torch.int64, device=device)


def graft_accept_compact(target_logits, tree_tok, tree_parent, tree_depth, Kc_ptrs, Vc_ptrs, Kt_ptrs, Vt_ptrs,
                         n_layers: int, Hkv: int, Lcap: int, L, out: Optional[dict] = None, status=None, ws=None,
                         stream=None, head_dim: int = HEAD_DIM, argmax=None, V: Optional[int] = None) -> dict:
    """target_logits [B][Kmax][V] f32, or None with ``argmax`` [B][Kmax] i32 given (and V)."""
    if target_logits is None:
        if argmax is None or V is None:
            raise ValueError("without target_logits pass argmax and V")
        B, Kmax = argmax.shape
        _need(argmax, "argmax", torch.int32, (B, Kmax))
    else:
        B, Kmax, V = target_logits.shape
        _need(target_logits, "target_logits", torch.float32)
    for name, t in (("tree_tok", tree_tok), ("tree_parent", tree_parent), ("tree_depth", tree_depth)):
        _need(t, name, torch.int32, (B, Kmax))
    _need(L, "L", torch.int32, (B,))
    for name, t in (("Kc_ptrs", Kc_ptrs), ("Vc_ptrs", Vc_ptrs), ("Kt_ptrs", Kt_ptrs), ("Vt_ptrs", Vt_ptrs)):
        _need(t, name, torch.int64, (n_layers,))
    dev = tree_tok.device
    if out is None:
        out = dict(argmax=argmax if argmax is not None else torch.empty(B, Kmax, dtype=torch.int32, device=dev),
                   acc_len=torch.empty(B, dtype=torch.int32, device=dev),
                   path=torch.empty(B, Kmax, dtype=torch.int32, device=dev),
                   out_tok=torch.empty(B, Kmax, dtype=torch.int32, device=dev),
                   bonus=torch.empty(B, dtype=torch.int32, device=dev))
    ws, nws = _ws(graft_accept_compact_workspace_size(B, Kmax, V), dev, ws)
    _check(lib().graft_accept_compact(B, Kmax, V, n_layers, _ptr(target_logits), _ptr(tree_tok), _ptr(tree_parent),
                                      _ptr(tree_depth), _ptr(Kc_ptrs), _ptr(Vc_ptrs), _ptr(Kt_ptrs), _ptr(Vt_ptrs),
                                      Hkv, head_dim, Lcap, _ptr(L), _ptr(out["argmax"]), _ptr(out["acc_len"]),
                                      _ptr(out["path"]), _ptr(out["out_tok"]), _ptr(out["bonus"]), _ptr(status),
                                      _ptr(ws), nws, _stream(stream)), "graft_accept_compact")
    return out


def graft_lm_head_argmax_workspace_size(N: int) -> int:
    n = _SZ()
    _check(lib().graft_lm_head_argmax_workspace_size(N, ctypes.byref(n)), "workspace size")
    return n.value


def graft_lm_head_argmax(H, W_lm, argmax=None, max_logit=None, status=None, ws=None, stream=None):
    """Greedy token per row of H [N][d] bf16 under the lm_head W_lm [V][d] bf16; returns (argmax, max_logit)."""
    N, d = H.shape
    V = W_lm.shape[0]
    _need(H, "H", torch.bfloat16, (N, d))
    _need(W_lm, "W_lm", torch.bfloat16, (V, d))
    dev = H.device
    if argmax is None:
        argmax = torch.empty(N, dtype=torch.int32, device=dev)
    if max_logit is None:
        max_logit = torch.empty(N, dtype=torch.float32, device=dev)
    ws, nws = _ws(graft_lm_head_argmax_workspace_size(N), dev, ws)
    _check(lib().graft_lm_head_argmax(N, d, V, _ptr(H), _ptr(W_lm), _ptr(argmax), _ptr(max_logit), _ptr(status),
                                      _ptr(ws), nws, _stream(stream)), "graft_lm_head_argmax")
    return argmax, max_logit


def graft_sample_tokens_workspace_size(B: int, Kmax: int, V: int) -> int:
    n = _SZ()
    _check(lib().graft_sample_tokens_workspace_size(B, Kmax, V, ctypes.byref(n)), "workspace size")
    return n.value


def graft_sample_tokens(target_logits, tree_pos, temperature: float, seed: int, sampled=None, ws=None, stream=None):
    """The target's sample per tree node (Gumbel-max with position-keyed Philox noise); [B][Kmax] int32."""
    B, Kmax, V = target_logits.shape
    _need(target_logits, "target_logits", torch.float32)
    _need(tree_pos, "tree_pos", torch.int32, (B, Kmax))
    if sampled is None:
        sampled = torch.empty(B, Kmax, dtype=torch.int32, device=target_logits.device)
    ws, nws = _ws(graft_sample_tokens_workspace_size(B, Kmax, V), target_logits.device, ws)
    _check(lib().graft_sample_tokens(B, Kmax, V, _ptr(target_logits), _ptr(tree_pos), float(temperature),
                                     int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(sampled), _ptr(ws), nws, _stream(stream)),
           "graft_sample_tokens")
    return sampled


def graft_lm_head_sample(H, W_lm, tree_pos, temperature: float, seed: int, sampled=None, status=None, ws=None,
                         stream=None):
    """graft_sample_tokens fused into the lm_head product; H [B*Kmax][d], tree_pos [B][Kmax]; returns [B*Kmax]."""
    N, d = H.shape
    V = W_lm.shape[0]
    _need(H, "H", torch.bfloat16, (N, d))
    _need(W_lm, "W_lm", torch.bfloat16, (V, d))
    B, Kmax = tree_pos.shape
    _need(tree_pos, "tree_pos", torch.int32, (B, Kmax))
    if B * Kmax != N:
        raise ValueError("H must have one row per tree node")
    if sampled is None:
        sampled = torch.empty(N, dtype=torch.int32, device=H.device)
    ws, nws = _ws(graft_lm_head_argmax_workspace_size(N), H.device, ws)
    _check(lib().graft_lm_head_sample(N, d, V, _ptr(H), _ptr(W_lm), Kmax, _ptr(tree_pos), float(temperature),
                                      int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(sampled), _ptr(status), _ptr(ws), nws,
                                      _stream(stream)), "graft_lm_head_sample")
    return sampled


def graft_update_M_workspace_size(n: int) -> int:
    sz = _SZ()
    _check(lib().graft_update_M_workspace_size(n, ctypes.byref(sz)), "workspace size")
    return sz.value


def graft_update_M(M_succ, M_cnt, src, dst, status=None, ws=None, stream=None):
    V, W = M_succ.shape
    _need(M_succ, "M_succ", torch.int32)
    _need(M_cnt, "M_cnt", torch.int32, (V, W))
    n = src.numel()
    _need(src, "src", torch.int32)
    _need(dst, "dst", torch.int32)
    if dst.numel() != n:
        raise ValueError("src and dst must have the same length")
    ws, nws = _ws(graft_update_M_workspace_size(n), M_succ.device, ws)
    _check(lib().graft_update_M(_ptr(M_succ), _ptr(M_cnt), V, W, _ptr(src), _ptr(dst), n, _ptr(status), _ptr(ws),
                                nws, _stream(stream)), "graft_update_M")


NOALLOC_MAX_PAIRS = 16384


def graft_update_M_noalloc(M_succ, M_cnt, src, dst, status=None, stream=None):
    """graft_update_M with the library's own fixed scratch (no workspace, nothing allocated).

    For callers that cannot provide device scratch memory; at most
    NOALLOC_MAX_PAIRS pairs per call, and calls that may overlap on the GPU
    must be ordered (they share one scratch array).
    """
    V, W = M_succ.shape
    _need(M_succ, "M_succ", torch.int32)
    _need(M_cnt, "M_cnt", torch.int32, (V, W))
    _need(src, "src", torch.int32)
    _need(dst, "dst", torch.int32)
    n = src.numel()
    if dst.numel() != n:
        raise ValueError("src and dst must have the same length")
    _check(lib().graft_update_M_noalloc(_ptr(M_succ), _ptr(M_cnt), V, W, _ptr(src), _ptr(dst), n, _ptr(status),
                                        _stream(stream)), "graft_update_M_noalloc")


def graft_status_string(code: int) -> str:
    return lib().graft_status_string(code).decode()


def graft_version() -> int:
    return lib().graft_version()


def graft_launch_count() -> int:
    return int(lib().graft_launch_count())


def graft_update_M_emitted_workspace_size(B: int, Kmax: int) -> int:
    n = _SZ()
    _check(lib().graft_update_M_emitted_workspace_size(B, Kmax, ctypes.byref(n)), "workspace size")
    return n.value


def graft_update_M_emitted(M_succ, M_cnt, tree_tok, out_tok, acc_len, status=None, ws=None, stream=None):
    """Add the bigrams of the tokens a step emitted (root -> out_tok[0] -> ... -> out_tok[acc_len-1])."""
    V, W = M_succ.shape
    _need(M_succ, "M_succ", torch.int32)
    _need(M_cnt, "M_cnt", torch.int32, (V, W))
    B, Kmax = tree_tok.shape
    _need(tree_tok, "tree_tok", torch.int32, (B, Kmax))
    _need(out_tok, "out_tok", torch.int32, (B, Kmax))
    _need(acc_len, "acc_len", torch.int32, (B,))
    ws, nws = _ws(graft_update_M_emitted_workspace_size(B, Kmax), M_succ.device, ws)
    _check(lib().graft_update_M_emitted(_ptr(M_succ), _ptr(M_cnt), V, W, B, Kmax, _ptr(tree_tok), _ptr(out_tok),
                                        _ptr(acc_len), _ptr(status), _ptr(ws), nws, _stream(stream)),
           "graft_update_M_emitted")


def graft_seed_M_from_tokens(M_succ, M_cnt, tokens, status=None, ws=None, stream=None):
    """Seed M with a prompt's bigrams (tokens[i] -> tokens[i+1]) in one order-independent update."""
    _need(tokens, "tokens", torch.int32)
    if tokens.numel() < 2:
        return
    t = tokens.reshape(-1)
    graft_update_M(M_succ, M_cnt, t[:-1], t[1:], status=status, ws=ws, stream=stream)
