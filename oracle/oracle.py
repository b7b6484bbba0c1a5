"""ctypes front end of the CPU oracle (oracle.cpp).

TEST INFRASTRUCTURE: only the test suite, the smoke check and the bench's CPU-baseline leg use this module. The
CUDA product path never imports it.

Arrays are numpy: bf16 tensors travel as their uint16 bit patterns, fp32 as float32; the oracle widens both exactly
to fp64. ``build()`` compiles oracle.cpp with g++ (fp64, no fast-math, no FMA contraction, OpenMP over requests).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path
from typing import Optional

import numpy as np

HERE = Path(__file__).resolve().parent
SRC = HERE / "oracle.cpp"
LIB = HERE / "liboracle.so"

F32, BF16 = 0, 1
ERRORS = {0: "ok", 1: "bad argument", 2: "NaN in logits", 3: "node budget exceeds the depth-limited tree",
          4: "not a valid draft tree"}


class OracleError(RuntimeError):
    pass


def compile_command(src=SRC, out=LIB):
    return ["g++", "-O2", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
            str(src), "-o", str(out)]


def build(force: bool = False, src=SRC, out=LIB) -> Path:
    out = Path(out)
    if force or not out.exists() or out.stat().st_mtime < Path(src).stat().st_mtime:
        tmp = out.with_suffix(f".{os.getpid()}.tmp.so")
        subprocess.run(compile_command(src, tmp), check=True)
        os.replace(tmp, out)
    return out


_P = ctypes.c_void_p
_I = ctypes.c_int
_D = ctypes.c_double


def load(path=None) -> ctypes.CDLL:
    lib = ctypes.CDLL(str(path or build()))
    lib.orc_topm.argtypes = [_P, _I, _I, _I, _I, _I, _P, _P, _I]
    lib.orc_lmhead_topm.argtypes = [_I, _I, _I, _I, _P, _I, _P, _I, _P, _P, _I]
    lib.orc_tree_attention.argtypes = [_I, _I, _I, _I, _I, _I, _P, _P, _P, _I, _P, _D, _P, _I]
    lib.orc_gru_step.argtypes = [_I, _I, _I, _P, _P, _P, _P, _P, _P, _P]
    lib.orc_child_logp.argtypes = [_I, _I, _P, _P, _P, _I, _D, _P, _P]
    lib.orc_build_trees.argtypes = [_I, _I, _I, _I, _I, _D, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P,
                                    _P, _P, _P, _P, _P, _P, _I]
    lib.orc_rescore.argtypes = [_I, _I, _I, _I, _I, _D, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P,
                                _P, _P, _P, _P, _I]
    lib.orc_build_trees_marginal.argtypes = [_I, _I, _I, _I, _I, _D, _P, _P, _P, _P, _P, _P, _P, _P, _I]
    lib.orc_build_trees_marginal.restype = _I
    lib.orc_accept_paths.argtypes = [_I, _I, _P, _P, _P, _P, _P, _P]
    lib.orc_accept_paths.restype = _I
    lib.orc_tree_size.argtypes = [_I, _I, ctypes.c_longlong]
    lib.orc_tree_size.restype = ctypes.c_longlong
    for f in (lib.orc_topm, lib.orc_gru_step, lib.orc_child_logp, lib.orc_build_trees, lib.orc_rescore):
        f.restype = _I
    return lib


_LIB: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = load()
    return _LIB


def _ptr(a: Optional[np.ndarray]):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    raise TypeError(f"oracle takes bf16 bit patterns (uint16) or float32, not {a.dtype}")


def _check(status: int):
    if status != 0:
        raise OracleError(ERRORS.get(status, f"status {status}"))


def topm(logits: np.ndarray, M: int, threads: int = 0, L=None):
    """logits [B,K,V] -> ids [B,K,M] int32, vals [B,K,M] float64."""
    L = L or lib()
    B, K, V = logits.shape
    logits = np.ascontiguousarray(logits)
    ids = np.empty((B, K, M), np.int32)
    vals = np.empty((B, K, M), np.float64)
    _check(L.orc_topm(_ptr(logits), _dtype_code(logits), B, K, V, M, _ptr(ids), _ptr(vals), threads))
    return ids, vals


def lmhead_topm(hidden: np.ndarray, w_head: np.ndarray, M: int, threads: int = 0, L=None):
    """hidden [R,D], w_head [V,D] (fp32, or bf16 bit patterns as uint16) -> ids [R,M] int32, vals [R,M] float64:
    the top-M of the full-vocabulary projection hidden @ w_head.T."""
    L = L or lib()
    R, D = hidden.shape
    V = w_head.shape[0]
    hidden = np.ascontiguousarray(hidden)
    w_head = np.ascontiguousarray(w_head)
    ids = np.empty((R, M), np.int32)
    vals = np.empty((R, M), np.float64)
    _check(L.orc_lmhead_topm(R, D, V, M, _ptr(hidden), _dtype_code(hidden), _ptr(w_head), _dtype_code(w_head),
                             _ptr(ids), _ptr(vals), threads))
    return ids, vals


def tree_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask: np.ndarray, scale: float, threads: int = 0,
                   L=None) -> np.ndarray:
    """q [B,n,Hq,d], k/v [B,Hkv,L+n,d] (fp32, or bf16 bit patterns as uint16), mask [B,n,n] uint8 -> out [B,n,Hq,d]
    float64: the verify pass's attention of each tree node over the prefix and its visible tree positions."""
    Lib = L or lib()
    B, n, Hq, d = q.shape
    Hkv, T = k.shape[1], k.shape[2]
    assert q.dtype == k.dtype == v.dtype
    out = np.empty((B, n, Hq, d), np.float64)
    _check(Lib.orc_tree_attention(B, n, T - n, Hq, Hkv, d, _ptr(np.ascontiguousarray(q)), _ptr(np.ascontiguousarray(k)),
                                  _ptr(np.ascontiguousarray(v)), _dtype_code(q),
                                  _ptr(np.ascontiguousarray(mask, np.uint8)), float(scale), _ptr(out), threads))
    return out


def gru_step(w_ih, w_hh, b_ih, b_hh, x: np.ndarray, h: np.ndarray, L=None) -> np.ndarray:
    L = L or lib()
    H = h.shape[0]
    E = x.shape[0]
    out = np.empty(H, np.float64)
    _check(L.orc_gru_step(H, E, _dtype_code(w_ih), _ptr(w_ih), _ptr(w_hh), _ptr(b_ih), _ptr(b_hh),
                          _ptr(np.ascontiguousarray(x, np.float64)), _ptr(np.ascontiguousarray(h, np.float64)),
                          _ptr(out)))
    return out


def child_logp(w_c, ids: np.ndarray, base: np.ndarray, T: float, h: np.ndarray, L=None) -> np.ndarray:
    L = L or lib()
    M = ids.shape[0]
    logp = np.empty(M, np.float64)
    _check(L.orc_child_logp(h.shape[0], _dtype_code(w_c), _ptr(w_c), _ptr(np.ascontiguousarray(ids, np.int32)),
                            _ptr(np.ascontiguousarray(base, np.float64)), M, float(T),
                            _ptr(np.ascontiguousarray(h, np.float64)), _ptr(logp)))
    return logp


def _weights_args(w: dict):
    return (_dtype_code(w["w_ih"]), _ptr(w["emb"]), _ptr(w["w_ih"]), _ptr(w["w_hh"]), _ptr(w.get("b_ih")),
            _ptr(w.get("b_hh")), _ptr(w["w_c"]))


def build_trees(ids, vals, h0, w: dict, n: int, max_depth: int, T: float, threads: int = 0, L=None) -> dict:
    """Best-first trees. ``w`` maps emb/w_ih/w_hh/b_ih/b_hh/w_c to host arrays (uint16 bits or float32)."""
    L = L or lib()
    B, K, M = ids.shape
    H = w["w_hh"].shape[1]
    E = w["w_ih"].shape[1]
    ids = np.ascontiguousarray(ids, np.int32)
    vals = np.ascontiguousarray(vals, np.float64)
    h0 = np.ascontiguousarray(h0, np.float64)
    out = dict(tokens=np.empty((B, n), np.int32), parents=np.empty((B, n), np.int32),
               depth=np.empty((B, n), np.int32), scores=np.empty((B, n), np.float64),
               mask=np.empty((B, n, n), np.uint8), gaps=np.empty((B, n), np.float64))
    wd, emb, wih, whh, bih, bhh, wc = _weights_args(w)
    _check(L.orc_build_trees(B, K, M, n, max_depth, float(T), _ptr(ids), _ptr(vals), _ptr(h0), H, E, wd, emb, wih,
                             whh, bih, bhh, wc, _ptr(out["tokens"]), _ptr(out["parents"]), _ptr(out["depth"]),
                             _ptr(out["scores"]), _ptr(out["mask"]), _ptr(out["gaps"]), threads))
    return out


def build_trees_marginal(ids, vals, n: int, max_depth: int, T: float, threads: int = 0, L=None) -> dict:
    """DDTree's factorised best-first trees from top-M candidates (no GRU, no correction)."""
    L = L or lib()
    B, K, M = ids.shape
    ids = np.ascontiguousarray(ids, np.int32)
    vals = np.ascontiguousarray(vals, np.float64)
    out = dict(tokens=np.empty((B, n), np.int32), parents=np.empty((B, n), np.int32),
               depth=np.empty((B, n), np.int32), scores=np.empty((B, n), np.float64),
               mask=np.empty((B, n, n), np.uint8), gaps=np.empty((B, n), np.float64))
    _check(L.orc_build_trees_marginal(B, K, M, n, max_depth, float(T), _ptr(ids), _ptr(vals), _ptr(out["tokens"]),
                                      _ptr(out["parents"]), _ptr(out["depth"]), _ptr(out["scores"]),
                                      _ptr(out["mask"]), _ptr(out["gaps"]), threads))
    return out


def accept_paths(tokens, parents, target_next, L=None) -> dict:
    """Accepted path of each verified tree: accept_len [B], path [B,n] (node indices, then -1), bonus [B]."""
    L = L or lib()
    B, n = tokens.shape
    tokens = np.ascontiguousarray(tokens, np.int32)
    parents = np.ascontiguousarray(parents, np.int32)
    target_next = np.ascontiguousarray(target_next, np.int32)
    assert target_next.shape == (B, n + 1)
    out = dict(accept_len=np.empty(B, np.int32), path=np.empty((B, n), np.int32), bonus=np.empty(B, np.int32))
    _check(L.orc_accept_paths(B, n, _ptr(tokens), _ptr(parents), _ptr(target_next), _ptr(out["accept_len"]),
                              _ptr(out["path"]), _ptr(out["bonus"])))
    return out


def rescore(ids, vals, h0, w: dict, tokens, parents, depth, max_depth: int, T: float, threads: int = 0,
            L=None) -> np.ndarray:
    """fp64 scores of given trees; raises OracleError if a tree is not a valid draft tree over the candidates."""
    L = L or lib()
    B, K, M = ids.shape
    n = tokens.shape[1]
    H = w["w_hh"].shape[1]
    E = w["w_ih"].shape[1]
    scores = np.empty((B, n), np.float64)
    wd, emb, wih, whh, bih, bhh, wc = _weights_args(w)
    _check(L.orc_rescore(B, K, M, n, max_depth, float(T), _ptr(np.ascontiguousarray(ids, np.int32)),
                         _ptr(np.ascontiguousarray(vals, np.float64)), _ptr(np.ascontiguousarray(h0, np.float64)),
                         H, E, wd, emb, wih, whh, bih, bhh, wc,
                         _ptr(np.ascontiguousarray(tokens, np.int32)), _ptr(np.ascontiguousarray(parents, np.int32)),
                         _ptr(np.ascontiguousarray(depth, np.int32)), _ptr(scores), threads))
    return scores


def tree_size(M: int, max_depth: int, cap: int = 1 << 62, L=None) -> int:
    return int((L or lib()).orc_tree_size(M, max_depth, cap))


def weights_of(inputs) -> dict:
    """Host arrays of a synth.Inputs' weights in storage form."""
    from speculative_decoding_tree_top_gb300.synth import host_array
    return {k: host_array(getattr(inputs, k)) for k in ("emb", "w_ih", "w_hh", "b_ih", "b_hh", "w_c")}


def round_(inputs, threads: int = 0, L=None) -> dict:
    """One whole round on the CPU: top-M, then the trees. Returns the tree dict plus 'ids' and 'vals'."""
    from speculative_decoding_tree_top_gb300.synth import host_array
    s = inputs.shape
    ids, vals = topm(host_array(inputs.logits), s.M, threads=threads, L=L)
    out = build_trees(ids, vals, host_array(inputs.h0).astype(np.float64), weights_of(inputs), s.n, s.max_depth,
                      s.T, threads=threads, L=L)
    out["ids"], out["vals"] = ids, vals
    return out
