"""Python binding of libdominotree (include/dominotree.h): argument marshalling only.

Every function here checks its torch tensors (device, dtype, shape, contiguity), passes their device pointers and
the current CUDA stream to the C ABI function of the same name, and raises DTError on a non-OK status. All the work
runs in the library's CUDA kernels; there is no fallback of any kind: without the compiled library the import of
``lib()`` fails loudly.
"""
from __future__ import annotations

import ctypes
import math
import enum
from dataclasses import dataclass
from typing import Optional

import torch

from . import buildlib


class Status(enum.IntEnum):
    OK = 0
    INVALID_ARG = 1
    UNSUPPORTED = 2
    CUDA = 3
    TIMEOUT = 4
    NUMERIC = 5


F32, BF16 = 0, 1


class DTError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = Status(status)
        super().__init__(f"{where}: {self.status.name} ({_LIB.dt_status_string(int(status)).decode() if _LIB else ''})")


class _Weights(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int), ("E", ctypes.c_int), ("dtype", ctypes.c_int), ("emb", ctypes.c_void_p),
                ("w_ih", ctypes.c_void_p), ("w_hh", ctypes.c_void_p), ("b_ih", ctypes.c_void_p),
                ("b_hh", ctypes.c_void_p), ("w_c", ctypes.c_void_p)]


_P, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_LIB: Optional[ctypes.CDLL] = None

# Every symbol the header declares, with its ctypes signature (restype, argtypes).
SIGNATURES = {
    "dt_workspace_init": (_I, [_P, _SZ, _P]),
    "dt_topm_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "dt_topm": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "dt_build_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "dt_build_trees": (_I, [_I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P, _P, ctypes.POINTER(_Weights), _P, _P,
                            _P, _P, _P, _P, _SZ, _P]),
    "dt_round": (_I, [_P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, ctypes.POINTER(_Weights), _P, _P, _P, _P,
                      _P, _P, _P, _P, _SZ, _P]),
    "dt_topm_static": (_I, [_P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "dt_accept_paths": (_I, [_I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "dt_build_trees_marginal": (_I, [_I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P, _P, _P, _P, _P, _P, _P, _SZ,
                                     _P]),
    "dt_lmhead_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "dt_lmhead_topm": (_I, [_I, _I, _I, _I, _P, _P, _I, _P, _P, _P, _SZ, _P]),
    "dt_tree_attention_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "dt_tree_attention": (_I, [_I, _I, _I, _I, _I, _I, _P, _P, _P, _I, _P, ctypes.c_float, _P, _P, _SZ, _P]),
    "dt_get_error": (_I, [_P, _P]),
    "dt_build_stats_read": (_I, [_P, _P, _P]),
    "dt_set_barrier_timeout_ns": (None, [ctypes.c_uint64]),
    "dt_set_lookahead": (_I, [_I]),
    "dt_set_topm_cluster": (_I, [_I]),
    "dt_status_string": (ctypes.c_char_p, [_I]),
    "dt_abi_version": (_I, []),
}


def lib() -> ctypes.CDLL:
    """The loaded library. Raises if it has not been built (``__graft_entry__.build()``)."""
    global _LIB
    if _LIB is None:
        if not buildlib.LIB.exists():
            raise RuntimeError(f"{buildlib.LIB} is missing: the CUDA library must be built first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(str(buildlib.LIB))
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def _check(status: int, where: str):
    if status != 0:
        raise DTError(status, where)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dev(t: torch.Tensor, name: str, dtype=None, shape=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, not {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, not {tuple(t.shape)}")
    return t.data_ptr()


def _code(dtype: torch.dtype) -> int:
    if dtype == torch.bfloat16:
        return BF16
    if dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {dtype}: bf16 or fp32")


def dt_topm_workspace_bytes(B: int, K: int, V: int, M: int) -> int:
    return int(lib().dt_topm_workspace_bytes(B, K, V, M))


def dt_build_workspace_bytes(B: int, K: int, V: int, M: int, n: int, H: int, E: int) -> int:
    """Workspace of a whole round (the top-M region, then the builder's own)."""
    return int(lib().dt_build_workspace_bytes(B, K, V, M, n, H, E))


def dt_workspace_init(workspace: torch.Tensor, stream=None):
    _check(lib().dt_workspace_init(_dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream)),
           "dt_workspace_init")


def new_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A zero-initialised workspace of at least ``nbytes`` bytes (a uint8 tensor)."""
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    dt_workspace_init(ws)
    return ws


def dt_get_error(workspace: torch.Tensor, stream=None) -> Status:
    return Status(lib().dt_get_error(_dev(workspace, "workspace", torch.uint8), _stream(stream)))


class _BuildStats(ctypes.Structure):
    _fields_ = [("launch_ns", ctypes.c_uint64), ("gather_ns", ctypes.c_uint64), ("gather_bytes", ctypes.c_uint64),
                ("waves", ctypes.c_int32), ("expansions", ctypes.c_int32)]


def dt_build_stats_read(workspace: torch.Tensor, stream=None) -> dict:
    """What the last dt_build_trees / dt_round launch on this workspace did (synchronises the stream)."""
    st = _BuildStats()
    _check(lib().dt_build_stats_read(_dev(workspace, "workspace", torch.uint8), ctypes.byref(st), _stream(stream)),
           "dt_build_stats_read")
    return {f: getattr(st, f) for f, _ in _BuildStats._fields_}


def dt_set_barrier_timeout_ns(ns: int):
    lib().dt_set_barrier_timeout_ns(int(ns))


def dt_set_lookahead(k: int):
    """Expansions per request per wave in dt_build_trees (0 = the library's choice); outputs do not depend on it."""
    _check(lib().dt_set_lookahead(int(k)), "dt_set_lookahead")


def dt_set_topm_cluster(enable: bool):
    """Whether small top-M launches run one thread-block cluster per row (the default); outputs do not depend on it."""
    _check(lib().dt_set_topm_cluster(int(bool(enable))), "dt_set_topm_cluster")


def dt_topm(logits: torch.Tensor, M: int, out_ids: Optional[torch.Tensor] = None,
            out_vals: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    """Top-M candidates of every row of logits [B,K,V] -> (ids [B,K,M] int32, vals [B,K,M] fp32)."""
    B, K, V = logits.shape
    if out_ids is None:
        out_ids = torch.empty((B, K, M), dtype=torch.int32, device=logits.device)
    if out_vals is None:
        out_vals = torch.empty((B, K, M), dtype=torch.float32, device=logits.device)
    if workspace is None:
        workspace = new_workspace(dt_topm_workspace_bytes(B, K, V, M), logits.device)
    _check(lib().dt_topm(_dev(logits, "logits"), _code(logits.dtype), B, K, V, M,
                         _dev(out_ids, "out_ids", torch.int32, (B, K, M)),
                         _dev(out_vals, "out_vals", torch.float32, (B, K, M)),
                         _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream)), "dt_topm")
    return out_ids, out_vals


def dt_lmhead_workspace_bytes(R: int, D: int, V: int, M: int) -> int:
    return int(lib().dt_lmhead_workspace_bytes(R, D, V, M))


def dt_lmhead_topm(hidden: torch.Tensor, w_head: torch.Tensor, M: int, out_ids: Optional[torch.Tensor] = None,
                   out_vals: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    """Top-M of the full-vocabulary projection hidden [R,D] . w_head [V,D]^T, fused (the logits are never written)
    -> (ids [R,M] int32, vals [R,M] fp32)."""
    R, D = hidden.shape
    V = w_head.shape[0]
    if out_ids is None:
        out_ids = torch.empty((R, M), dtype=torch.int32, device=hidden.device)
    if out_vals is None:
        out_vals = torch.empty((R, M), dtype=torch.float32, device=hidden.device)
    if workspace is None:
        workspace = new_workspace(dt_lmhead_workspace_bytes(R, D, V, M), hidden.device)
    _check(lib().dt_lmhead_topm(R, D, V, M, _dev(hidden, "hidden", hidden.dtype, (R, D)),
                                _dev(w_head, "w_head", hidden.dtype, (V, D)), _code(hidden.dtype),
                                _dev(out_ids, "out_ids", torch.int32, (R, M)),
                                _dev(out_vals, "out_vals", torch.float32, (R, M)),
                                _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream)),
           "dt_lmhead_topm")
    return out_ids, out_vals


def dt_tree_attention_workspace_bytes(B: int, n: int, L: int, Hq: int, Hkv: int, d: int) -> int:
    return int(lib().dt_tree_attention_workspace_bytes(B, n, L, Hq, Hkv, d))


def dt_tree_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, mask: torch.Tensor, scale: float,
                      out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, stream=None):
    """The verify pass's tree attention: q [B,n,Hq,d], k/v [B,Hkv,L+n,d] (bf16), mask [B,n,n] uint8
    -> out [B,n,Hq,d] fp32."""
    B, n, Hq, d = q.shape
    Hkv, T = k.shape[1], k.shape[2]
    L = T - n
    if out is None:
        out = torch.empty((B, n, Hq, d), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = new_workspace(dt_tree_attention_workspace_bytes(B, n, L, Hq, Hkv, d), q.device)
    _check(lib().dt_tree_attention(B, n, L, Hq, Hkv, d, _dev(q, "q", q.dtype, (B, n, Hq, d)),
                                   _dev(k, "k", q.dtype, (B, Hkv, T, d)), _dev(v, "v", q.dtype, (B, Hkv, T, d)),
                                   _code(q.dtype), _dev(mask, "mask", torch.uint8, (B, n, n)), float(scale),
                                   _dev(out, "out", torch.float32, (B, n, Hq, d)),
                                   _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream)),
           "dt_tree_attention")
    return out


def dt_topm_static(logits: torch.Tensor, M: int, out_ids: Optional[torch.Tensor] = None,
                   out_vals: Optional[torch.Tensor] = None, stream=None):
    """dt_topm without a workspace: the library's fixed device scratch array instead (see dominotree.h)."""
    B, K, V = logits.shape
    if out_ids is None:
        out_ids = torch.empty((B, K, M), dtype=torch.int32, device=logits.device)
    if out_vals is None:
        out_vals = torch.empty((B, K, M), dtype=torch.float32, device=logits.device)
    _check(lib().dt_topm_static(_dev(logits, "logits"), _code(logits.dtype), B, K, V, M,
                                _dev(out_ids, "out_ids", torch.int32, (B, K, M)),
                                _dev(out_vals, "out_vals", torch.float32, (B, K, M)), _stream(stream)),
           "dt_topm_static")
    return out_ids, out_vals


@dataclass
class Weights:
    """The drafter's correction weights (shared by all requests): GRU (gate rows r|z|n), embeddings, W_c."""
    emb: torch.Tensor                 # [V,E]
    w_ih: torch.Tensor                # [3H,E]
    w_hh: torch.Tensor                # [3H,H]
    b_ih: Optional[torch.Tensor]      # [3H] or None
    b_hh: Optional[torch.Tensor]      # [3H] or None
    w_c: torch.Tensor                 # [V,H]

    @property
    def H(self) -> int:
        return self.w_hh.shape[1]

    @property
    def E(self) -> int:
        return self.w_ih.shape[1]

    def struct(self) -> _Weights:
        dt = self.w_ih.dtype
        H, E, V = self.H, self.E, self.emb.shape[0]
        opt = lambda t, n: _dev(t, n, dt, (3 * H,)) if t is not None else None
        return _Weights(H, E, _code(dt), _dev(self.emb, "emb", dt, (V, E)), _dev(self.w_ih, "w_ih", dt, (3 * H, E)),
                        _dev(self.w_hh, "w_hh", dt, (3 * H, H)), opt(self.b_ih, "b_ih"), opt(self.b_hh, "b_hh"),
                        _dev(self.w_c, "w_c", dt, (V, H)))

    @classmethod
    def of(cls, inputs) -> "Weights":
        return cls(inputs.emb, inputs.w_ih, inputs.w_hh, inputs.b_ih, inputs.b_hh, inputs.w_c)


def dt_build_trees(topm_ids: torch.Tensor, topm_vals: torch.Tensor, h0: torch.Tensor, weights: Weights, n: int,
                   max_depth: int, T: float, out: Optional[dict] = None, workspace: Optional[torch.Tensor] = None,
                   stream=None) -> dict:
    """Best-first conditional trees -> dict of tokens/parents/depth [B,n] int32, scores [B,n] fp32,
    mask [B,n,n] uint8."""
    B, K, M = topm_ids.shape
    V = weights.emb.shape[0]
    dev = topm_ids.device
    if out is None:
        out = alloc_tree_outputs(B, n, dev)
    if workspace is None:
        workspace = new_workspace(dt_build_workspace_bytes(B, K, V, M, n, weights.H, weights.E), dev)
    w = weights.struct()
    _check(lib().dt_build_trees(
        B, K, V, M, n, max_depth, float(T), _dev(topm_ids, "topm_ids", torch.int32, (B, K, M)),
        _dev(topm_vals, "topm_vals", torch.float32, (B, K, M)), _dev(h0, "h0", torch.float32, (B, weights.H)),
        ctypes.byref(w), _dev(out["tokens"], "out_tokens", torch.int32, (B, n)),
        _dev(out["parents"], "out_parents", torch.int32, (B, n)), _dev(out["depth"], "out_depth", torch.int32, (B, n)),
        _dev(out["scores"], "out_scores", torch.float32, (B, n)),
        _dev(out["mask"], "out_mask", torch.uint8, (B, n, n)), _dev(workspace, "workspace", torch.uint8),
        workspace.numel(), _stream(stream)), "dt_build_trees")
    return out


def dt_round(logits: torch.Tensor, h0: torch.Tensor, weights: Weights, M: int, n: int, max_depth: int, T: float,
             topm_ids: Optional[torch.Tensor] = None, topm_vals: Optional[torch.Tensor] = None,
             out: Optional[dict] = None, workspace: Optional[torch.Tensor] = None, stream=None) -> dict:
    """dt_topm then dt_build_trees in one call, every argument checked before either launch -> the tree outputs of
    dt_build_trees; the candidates land in ``topm_ids`` / ``topm_vals`` [B,K,M]."""
    B, K, V = logits.shape
    dev = logits.device
    if topm_ids is None:
        topm_ids = torch.empty((B, K, M), dtype=torch.int32, device=dev)
    if topm_vals is None:
        topm_vals = torch.empty((B, K, M), dtype=torch.float32, device=dev)
    if out is None:
        out = alloc_tree_outputs(B, n, dev)
    if workspace is None:
        workspace = new_workspace(dt_build_workspace_bytes(B, K, V, M, n, weights.H, weights.E), dev)
    w = weights.struct()
    _check(lib().dt_round(
        _dev(logits, "logits"), _code(logits.dtype), B, K, V, M, n, max_depth, float(T),
        _dev(h0, "h0", torch.float32, (B, weights.H)), ctypes.byref(w),
        _dev(topm_ids, "topm_ids", torch.int32, (B, K, M)), _dev(topm_vals, "topm_vals", torch.float32, (B, K, M)),
        _dev(out["tokens"], "out_tokens", torch.int32, (B, n)), _dev(out["parents"], "out_parents", torch.int32, (B, n)),
        _dev(out["depth"], "out_depth", torch.int32, (B, n)), _dev(out["scores"], "out_scores", torch.float32, (B, n)),
        _dev(out["mask"], "out_mask", torch.uint8, (B, n, n)), _dev(workspace, "workspace", torch.uint8),
        workspace.numel(), _stream(stream)), "dt_round")
    return out


def dt_build_trees_marginal(topm_ids: torch.Tensor, topm_vals: torch.Tensor, V: int, n: int, max_depth: int,
                            T: float, out: Optional[dict] = None, workspace: Optional[torch.Tensor] = None,
                            stream=None) -> dict:
    """DDTree's factorised best-first trees (no GRU, no correction) -> the same outputs as dt_build_trees."""
    B, K, M = topm_ids.shape
    dev = topm_ids.device
    if out is None:
        out = alloc_tree_outputs(B, n, dev)
    if workspace is None:
        workspace = new_workspace(256, dev)
    _check(lib().dt_build_trees_marginal(
        B, K, V, M, n, max_depth, float(T), _dev(topm_ids, "topm_ids", torch.int32, (B, K, M)),
        _dev(topm_vals, "topm_vals", torch.float32, (B, K, M)), _dev(out["tokens"], "out_tokens", torch.int32, (B, n)),
        _dev(out["parents"], "out_parents", torch.int32, (B, n)), _dev(out["depth"], "out_depth", torch.int32, (B, n)),
        _dev(out["scores"], "out_scores", torch.float32, (B, n)),
        _dev(out["mask"], "out_mask", torch.uint8, (B, n, n)), _dev(workspace, "workspace", torch.uint8),
        workspace.numel(), _stream(stream)), "dt_build_trees_marginal")
    return out


def dt_accept_paths(tokens: torch.Tensor, parents: torch.Tensor, target_next: torch.Tensor, out: Optional[dict] = None,
                    stream=None) -> dict:
    """Accepted path of each verified tree -> accept_len [B], path [B,n] (node indices, then -1), bonus [B]."""
    B, n = tokens.shape
    dev = tokens.device
    if out is None:
        out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                   path=torch.empty((B, n), dtype=torch.int32, device=dev),
                   bonus=torch.empty(B, dtype=torch.int32, device=dev))
    _check(lib().dt_accept_paths(B, n, _dev(tokens, "tokens", torch.int32, (B, n)),
                                 _dev(parents, "parents", torch.int32, (B, n)),
                                 _dev(target_next, "target_next", torch.int32, (B, n + 1)),
                                 _dev(out["accept_len"], "out_accept_len", torch.int32, (B,)),
                                 _dev(out["path"], "out_path", torch.int32, (B, n)),
                                 _dev(out["bonus"], "out_bonus", torch.int32, (B,)), _stream(stream)),
           "dt_accept_paths")
    return out


def alloc_tree_outputs(B: int, n: int, device) -> dict:
    return dict(tokens=torch.empty((B, n), dtype=torch.int32, device=device),
                parents=torch.empty((B, n), dtype=torch.int32, device=device),
                depth=torch.empty((B, n), dtype=torch.int32, device=device),
                scores=torch.empty((B, n), dtype=torch.float32, device=device),
                mask=torch.empty((B, n, n), dtype=torch.uint8, device=device))


class Round:
    """Preallocated buffers for one drafting round of a fixed shape: dt_topm then dt_build_trees on one stream."""

    def __init__(self, B, K, V, M, n, max_depth, T, weights: Weights, device="cuda"):
        self.B, self.K, self.V, self.M, self.n, self.max_depth, self.T = B, K, V, M, n, max_depth, T
        self.weights = weights
        self.ids = torch.empty((B, K, M), dtype=torch.int32, device=device)
        self.vals = torch.empty((B, K, M), dtype=torch.float32, device=device)
        self.out = alloc_tree_outputs(B, n, device)
        self.workspace = new_workspace(dt_build_workspace_bytes(B, K, V, M, n, weights.H, weights.E), device)

        self._topm_key = self._build_key = None

    def topm(self, logits: torch.Tensor, stream=None):
        """dt_topm into this round's ids/vals. The marshalled arguments are kept while the logits tensor (address,
        shape, dtype) and the stream stay the same, so a repeated call costs one C call."""
        st = _stream(stream)
        key = (logits.data_ptr(), tuple(logits.shape), logits.dtype, st)
        if key != self._topm_key:
            B, K, V = logits.shape
            if (B, K, V) != (self.B, self.K, self.V):
                raise ValueError(f"logits must have shape {(self.B, self.K, self.V)}, not {(B, K, V)}")
            self._topm_args = (_dev(logits, "logits"), _code(logits.dtype), B, K, V, self.M,
                               _dev(self.ids, "out_ids"), _dev(self.vals, "out_vals"),
                               _dev(self.workspace, "workspace", torch.uint8), self.workspace.numel(), st)
            self._topm_key = key
        _check(lib().dt_topm(*self._topm_args), "dt_topm")
        return self.ids, self.vals

    def build(self, h0: torch.Tensor, stream=None) -> dict:
        """dt_build_trees from this round's ids/vals into its outputs (arguments kept like ``topm``'s, also keyed
        by the weights' tensors)."""
        st = _stream(stream)
        w = self.weights
        key = (h0.data_ptr(), tuple(h0.shape), h0.dtype, st, id(w),
               *(t.data_ptr() if t is not None else 0 for t in (w.emb, w.w_ih, w.w_hh, w.b_ih, w.b_hh, w.w_c)))
        if key != self._build_key:
            self._wstruct = w.struct()
            o = self.out
            self._build_args = (
                self.B, self.K, self.V, self.M, self.n, self.max_depth, float(self.T), _dev(self.ids, "topm_ids"),
                _dev(self.vals, "topm_vals"), _dev(h0, "h0", torch.float32, (self.B, w.H)),
                ctypes.byref(self._wstruct), _dev(o["tokens"], "out_tokens"), _dev(o["parents"], "out_parents"),
                _dev(o["depth"], "out_depth"), _dev(o["scores"], "out_scores"), _dev(o["mask"], "out_mask"),
                _dev(self.workspace, "workspace", torch.uint8), self.workspace.numel(), st)
            self._build_key = key
        _check(lib().dt_build_trees(*self._build_args), "dt_build_trees")
        return self.out

    def build_marginal(self, stream=None) -> dict:
        """dt_build_trees_marginal (DDTree's factorised scoring) from this round's ids/vals into its outputs."""
        st = _stream(stream)
        if getattr(self, "_marg_key", None) != st:
            o = self.out
            self._marg_args = (self.B, self.K, self.V, self.M, self.n, self.max_depth, float(self.T),
                               _dev(self.ids, "topm_ids"), _dev(self.vals, "topm_vals"), _dev(o["tokens"], "out_tokens"),
                               _dev(o["parents"], "out_parents"), _dev(o["depth"], "out_depth"),
                               _dev(o["scores"], "out_scores"), _dev(o["mask"], "out_mask"),
                               _dev(self.workspace, "workspace", torch.uint8), self.workspace.numel(), st)
            self._marg_key = st
        _check(lib().dt_build_trees_marginal(*self._marg_args), "dt_build_trees_marginal")
        return self.out

    def round(self, logits: torch.Tensor, h0: torch.Tensor, stream=None) -> dict:
        """dt_round: the top-M into this round's ids/vals and the tree into its outputs, in one call (arguments kept
        like ``topm``'s)."""
        st = _stream(stream)
        w = self.weights
        key = (logits.data_ptr(), tuple(logits.shape), logits.dtype, h0.data_ptr(), tuple(h0.shape), h0.dtype, st,
               id(w), *(t.data_ptr() if t is not None else 0 for t in (w.emb, w.w_ih, w.w_hh, w.b_ih, w.b_hh, w.w_c)))
        if key != getattr(self, "_round_key", None):
            B, K, V = logits.shape
            if (B, K, V) != (self.B, self.K, self.V):
                raise ValueError(f"logits must have shape {(self.B, self.K, self.V)}, not {(B, K, V)}")
            self._round_w = w.struct()
            o = self.out
            self._round_args = (
                _dev(logits, "logits"), _code(logits.dtype), B, K, V, self.M, self.n, self.max_depth, float(self.T),
                _dev(h0, "h0", torch.float32, (self.B, w.H)), ctypes.byref(self._round_w), _dev(self.ids, "topm_ids"),
                _dev(self.vals, "topm_vals"), _dev(o["tokens"], "out_tokens"), _dev(o["parents"], "out_parents"),
                _dev(o["depth"], "out_depth"), _dev(o["scores"], "out_scores"), _dev(o["mask"], "out_mask"),
                _dev(self.workspace, "workspace", torch.uint8), self.workspace.numel(), st)
            self._round_key = key
        _check(lib().dt_round(*self._round_args), "dt_round")
        return self.out

    def capture(self, logits: torch.Tensor, h0: torch.Tensor) -> torch.cuda.CUDAGraph:
        """One dt_round call on these tensors, captured as a CUDA graph (its two launches, the cluster top-M and the
        cooperative builder, as graph nodes). ``replay()`` reruns the round on whatever ``logits`` and ``h0`` then
        hold, into this round's ids/vals and outputs, without the per-launch host work. The addresses are fixed at
        capture: new inputs go into the same tensors."""
        side = torch.cuda.Stream(device=self.workspace.device)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.round(logits, h0)  # marshalled for the capture stream; the library's one-time set-up done
        side.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            self.round(logits, h0)
        torch.cuda.current_stream().wait_stream(side)
        return g

    def __call__(self, logits: torch.Tensor, h0: torch.Tensor, stream=None) -> dict:
        return self.round(logits, h0, stream)

    def check(self, stream=None):
        _check(int(dt_get_error(self.workspace, stream)), "device status")


def packed_buffers(specs, device, pin: bool = False):
    """One byte buffer holding several tensors, each starting on a 16-byte boundary: ``specs`` is a list of (name,
    shape, dtype). Returns the buffer and a dict of views into it. One copy of the buffer moves them all."""
    offs, o = [], 0
    for _, shape, dtype in specs:
        nbytes = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        offs.append((o, nbytes))
        o += (nbytes + 15) // 16 * 16
    if pin:
        buf = torch.empty(o, dtype=torch.uint8, device="cpu", pin_memory=True)
    else:
        buf = torch.empty(o, dtype=torch.uint8, device=device)
    views = {name: buf[off:off + nb].view(dtype).view(shape) for (name, shape, dtype), (off, nb) in zip(specs, offs)}
    return buf, views


class HostRound(Round):
    """A round whose inputs and outputs live in pinned host memory: each call copies the logits and h0 to the device
    (one copy: they sit in one buffer), runs dt_round (dt_topm and dt_build_trees), and copies the tree back (one
    copy of one buffer), all on one stream. The caller writes a round's inputs into ``host_logits`` / ``host_h0``."""

    def __init__(self, B, K, V, M, n, max_depth, T, weights: Weights, logits_dtype, device="cuda"):
        super().__init__(B, K, V, M, n, max_depth, T, weights, device)
        ins = [("logits", (B, K, V), logits_dtype), ("h0", (B, weights.H), torch.float32)]
        self._din, d = packed_buffers(ins, device)
        self._hin, h = packed_buffers(ins, device, pin=True)
        self.d_logits, self.d_h0 = d["logits"], d["h0"]
        self.host_logits, self.host_h0 = h["logits"], h["h0"]
        outs = [("tokens", (B, n), torch.int32), ("parents", (B, n), torch.int32), ("depth", (B, n), torch.int32),
                ("scores", (B, n), torch.float32), ("mask", (B, n, n), torch.uint8)]
        self._dout, self.out = packed_buffers(outs, device)
        self._hout, self.host_out = packed_buffers(outs, device, pin=True)

    def h2d_bytes(self) -> int:
        return self._hin.numel()

    def d2h_bytes(self) -> int:
        return self._hout.numel()

    def run(self, host_logits: Optional[torch.Tensor] = None, host_h0: Optional[torch.Tensor] = None,
            stream=None) -> dict:
        """One round from the pinned inputs. Tensors passed here are first copied into them on the host."""
        if host_logits is not None:
            self.host_logits.copy_(host_logits)
        if host_h0 is not None:
            self.host_h0.copy_(host_h0)
        self._din.copy_(self._hin, non_blocking=True)
        self(self.d_logits, self.d_h0, stream)
        self._hout.copy_(self._dout, non_blocking=True)
        return self.host_out

    def capture(self) -> torch.cuda.CUDAGraph:
        """``run()`` captured as a CUDA graph: the copy in, the round's two launches and the copy out as graph nodes.
        ``replay()`` then runs a round on whatever ``host_logits`` / ``host_h0`` hold and leaves its tree in
        ``host_out`` once the stream has been synchronised."""
        side = torch.cuda.Stream(device=self.workspace.device)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.run()  # marshalled for the capture stream
        side.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            self.run()
        torch.cuda.current_stream().wait_stream(side)
        return g
