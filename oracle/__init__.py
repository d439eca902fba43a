"""ctypes front end of the fp64 CPU oracle (oracle.cpp).

Test infrastructure only: imported by tests/, by the package smoke check and
by the benchmark's CPU-baseline leg.  The product path never imports it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with the host C++ compiler (no vendor code involved)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


class _Out(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "accept_len", "num_out", "out_tokens", "bonus", "accept_rows", "commit_cu",
        "commit_src_slot", "commit_dst_pos", "status", "min_gap", "test_gap", "draw_gap")]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I32, I64, D = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.oracle_verify_chain.argtypes = [ctypes.c_int, P, ctypes.c_int, I64, I32, I64, I32, I32, P, P, P,
                                                I64, P, P, P, P, P, ctypes.POINTER(_Out), I32]
            lib.oracle_verify_tree.argtypes = [ctypes.c_int, P, ctypes.c_int, I64, I32, I32, I32, P, P, P, P, P,
                                               D, D, P, P, P, P, ctypes.POINTER(_Out), I32]
            lib.oracle_row_stats.argtypes = [P, ctypes.c_int, I64, I64, I32, P, P, P, P, P, P, P]
            lib.oracle_row_probs.argtypes = [P, ctypes.c_int, I64, I64, I32, D, P]
            lib.oracle_residual.argtypes = [P, P, I64, P]
            lib.oracle_accept.argtypes = [D, D, D]
            lib.oracle_accept.restype = ctypes.c_int
            lib.oracle_sample_index.argtypes = [P, I64, D, ctypes.POINTER(ctypes.c_double)]
            lib.oracle_sample_index.restype = I64
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def _dtype_code(dtype: str) -> int:
    return {"f32": 0, "bf16": 1}[dtype]


def _alloc_out(batch: int, max_len: int, rows: int) -> dict:
    return {
        "accept_len": np.zeros(batch, np.int32),
        "num_out": np.zeros(batch, np.int32),
        "out_tokens": np.zeros((batch, max_len), np.int32),
        "bonus": np.zeros(batch, np.int32),
        "accept_rows": np.zeros((batch, max_len), np.int32),
        "commit_cu": np.zeros(batch + 1, np.int32),
        "commit_src_slot": np.full(max(rows, 1), -1, np.int64),
        "commit_dst_pos": np.full(max(rows, 1), -1, np.int64),
        "status": np.zeros(batch, np.uint32),
        "min_gap": np.zeros(batch, np.float64),
        "test_gap": np.zeros((batch, max_len), np.float64),  # per step: gap of the acceptance test(s) made there
        "draw_gap": np.zeros(batch, np.float64),             # gap of the final draw
    }


def _out_struct(o: dict) -> _Out:
    return _Out(*[o[n].ctypes.data for n, _ in _Out._fields_])


def verify_chain(w, greedy_all: bool = False, threads: int = 1, cu_seqlens=None, batch=None) -> dict:
    """Oracle outputs for a chain / ragged workload (greedy_all: every request greedy)."""
    lib = _load()
    logits = np.ascontiguousarray(w.logits)
    cu = _c(w.cu_seqlens if cu_seqlens is None else cu_seqlens, np.int32)
    B = w.batch if batch is None else batch
    ids = _c(w.verify_ids, np.int32)
    q = None if greedy_all else _c(w.q, np.float32)
    T = None if greedy_all else _c(w.temperature, np.float32)
    ua = None if greedy_all else _c(w.u_accept, np.float32)
    uf = None if greedy_all else _c(w.u_final, np.float32)
    slots, sl = _c(w.row_slots, np.int64), _c(w.seq_lens, np.int64)
    o = _alloc_out(B, w.max_len, w.rows)
    st = _out_struct(o)
    lib.oracle_verify_chain(1 if greedy_all else 0, _p(logits), _dtype_code(w.dtype), w.vocab, B, w.rows,
                            w.max_len, w.vocab, _p(cu), _p(ids), _p(q), w.vocab, _p(T), _p(ua), _p(uf),
                            _p(slots), _p(sl), ctypes.byref(st), threads)
    return o


def scatter_candidates(cand_ids, cand_probs, vocab: int):
    """Dense q from candidate lists, [E2D] §6.5: the selector's sparse q is
    scattered into vocabulary coordinates (zero elsewhere) before rejection.

    Returns (q [R, vocab] float32, bad [R] bool).  Id -1 is padding; any other
    id outside [0, vocab) is left out of q and marks its row bad.  Repeated ids
    add up (accumulated in fp64).
    """
    ids = np.asarray(cand_ids, dtype=np.int64)
    pr = np.asarray(cand_probs, dtype=np.float64)
    R, K = ids.shape
    ok = (ids >= 0) & (ids < vocab)
    bad = np.any((ids != -1) & ~ok, axis=1)
    q = np.zeros((R, vocab), dtype=np.float64)
    rr = np.repeat(np.arange(R), K).reshape(R, K)
    np.add.at(q, (rr[ok], ids[ok]), pr[ok])
    return q.astype(np.float32), bad


def verify_chain_sparse(w, threads: int = 1) -> dict:
    """Oracle outputs for a chain whose q is given as candidate lists: the
    dense chain verification over the scattered q.  A request is flagged
    SV_DEV_TOKEN_RANGE (bit 1) when a tested row (every row but its last) has a
    candidate id outside [0, vocab) other than the padding -1."""
    import dataclasses
    q, bad = scatter_candidates(w.cand_ids, w.cand_probs, w.vocab)
    dense = dataclasses.replace(w, q=q, kind="rejection_chain")
    o = verify_chain(dense, threads=threads)
    cu = np.asarray(w.cu_seqlens, dtype=np.int64)
    for b in range(len(cu) - 1):
        if cu[b + 1] - 1 > cu[b] and bad[cu[b]:cu[b + 1] - 1].any():
            o["status"][b] |= np.uint32(1)
    return o


def verify_tree(w, mode: str, threads: int = 1, use_lists: bool = False) -> dict:
    """Oracle outputs for a tree workload; mode 'greedy' or 'target_only'."""
    lib = _load()
    logits = np.ascontiguousarray(w.logits)
    tok, par = _c(w.tokens, np.int32), _c(w.parents, np.int32)
    fc = _c(w.first_child, np.int32) if use_lists else None
    ns = _c(w.next_sibling, np.int32) if use_lists else None
    sampling = mode == "target_only"
    T = _c(w.temperature, np.float32) if sampling else None
    ua = _c(w.u_accept, np.float32) if sampling else None
    uf = _c(w.u_final, np.float32) if sampling else None
    slots, sl = _c(w.row_slots, np.int64), _c(w.seq_lens, np.int64)
    o = _alloc_out(w.batch, w.nodes, w.rows)
    st = _out_struct(o)
    lib.oracle_verify_tree(1 if sampling else 0, _p(logits), _dtype_code(w.dtype), w.vocab, w.batch, w.nodes,
                           w.vocab, _p(tok), _p(par), _p(fc), _p(ns), _p(T), float(w.threshold_single),
                           float(w.threshold_acc), _p(ua), _p(uf), _p(slots), _p(sl), ctypes.byref(st), threads)
    return o


def row_stats(logits: np.ndarray, dtype: str, row_temp=None, probe=None) -> dict:
    lib = _load()
    logits = np.ascontiguousarray(logits)
    R, V = logits.shape
    out = {"max": np.zeros(R), "argmax": np.zeros(R, np.int32), "z": np.zeros(R), "p": np.zeros(R),
           "flags": np.zeros(R, np.uint32)}
    rt, pr = _c(row_temp, np.float32), _c(probe, np.int32)
    lib.oracle_row_stats(_p(logits), _dtype_code(dtype), V, R, V, _p(rt), _p(pr), _p(out["max"]),
                         _p(out["argmax"]), _p(out["z"]), _p(out["p"]), _p(out["flags"]))
    return out


def row_probs(logits: np.ndarray, dtype: str, row: int, T: float) -> np.ndarray:
    lib = _load()
    logits = np.ascontiguousarray(logits)
    R, V = logits.shape
    p = np.zeros(V)
    rc = lib.oracle_row_probs(_p(logits), _dtype_code(dtype), V, row, V, float(T), _p(p))
    if rc != 0:
        raise ValueError("row has no usable maximum or T <= 0")
    return p


def residual(p: np.ndarray, q: np.ndarray) -> np.ndarray:
    lib = _load()
    p = np.ascontiguousarray(p, np.float64)
    q = np.ascontiguousarray(q, np.float32)
    w = np.zeros_like(p)
    lib.oracle_residual(_p(p), _p(q), len(p), _p(w))
    return w


def accept(p: float, q: float, u: float) -> bool:
    return bool(_load().oracle_accept(float(p), float(q), float(u)))


def sample_index(w: np.ndarray, u: float) -> tuple:
    lib = _load()
    w = np.ascontiguousarray(w, np.float64)
    g = ctypes.c_double(0.0)
    v = lib.oracle_sample_index(_p(w), len(w), float(u), ctypes.byref(g))
    return int(v), g.value
