"""Python binding of libspecverify (ctypes; argument marshalling only).

Every step of the verification runs in the CUDA library; this module only
turns torch tensors into device pointers and sizes, calls the C ABI declared
in include/specverify.h on the current torch stream, and raises on a bad
status.  The library must be built (reject_row_vocab_gb300._build.build());
importing this module without it raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libspecverify.so")

SV_F32, SV_BF16 = 0, 1
STATUS = {0: "SV_OK", 1: "SV_ERR_NULL_ARG", 2: "SV_ERR_BAD_SHAPE", 3: "SV_ERR_BAD_DTYPE", 4: "SV_ERR_MISALIGNED",
          5: "SV_ERR_UNSUPPORTED", 6: "SV_ERR_WORKSPACE_TOO_SMALL", 7: "SV_ERR_CUDA"}
DEV_TOKEN_RANGE, DEV_NONFINITE, DEV_BAD_TREE, DEV_BAD_LAYOUT, DEV_RESIDUAL_EMPTY, DEV_DUP_SIBLING = 1, 2, 4, 8, 16, 32

ENTRY_POINTS = ("spec_verify_workspace_bytes", "spec_verify_status_string", "spec_verify_greedy_chain",
                "spec_verify_greedy_tree", "spec_verify_rejection_chain", "spec_verify_rejection_ragged",
                "spec_verify_target_only_tree", "spec_verify_row_stats", "spec_verify_set_stats_events",
                "spec_verify_last_cuda_error", "spec_verify_rejection_chain_noalloc",
                "spec_verify_dspark_workspace_bytes", "spec_verify_dspark_budget", "spec_verify_dspark_verify_lens",
                "spec_verify_sparse_workspace_bytes", "spec_verify_rejection_chain_sparse", "spec_verify_build_tree",
                "spec_verify_sample_match_chain")


class SpecVerifyError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__("%s returned %s (%d): %s" % (fn, STATUS.get(code, "?"), code, msg))
        self.code = code


class SvOut(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "accept_len", "num_out", "out_tokens", "bonus", "accept_rows", "commit_cu", "commit_src_slot",
        "commit_dst_pos", "dev_status")]


_lib = None


def load_library():
    """Load libspecverify.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libspecverify.so is not built (%s); run reject_row_vocab_gb300._build.build()" % LIB_PATH)
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, F, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    OUT = ctypes.POINTER(SvOut)
    sig = {
        "spec_verify_workspace_bytes": ([I64, I32, I32, I32], SZ),
        "spec_verify_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "spec_verify_last_cuda_error": ([], ctypes.c_char_p),
        "spec_verify_greedy_chain": ([P, ctypes.c_int, I64, I32, I32, I32, P, P, P, OUT, P, SZ, P], ctypes.c_int),
        "spec_verify_greedy_tree": ([P, ctypes.c_int, I64, I32, I32, I32, P, P, P, P, P, P, OUT, P, SZ, P],
                                    ctypes.c_int),
        "spec_verify_rejection_chain": ([P, ctypes.c_int, I64, I32, I32, I32, P, P, I64, P, P, P, P, P, OUT, P, SZ,
                                         P], ctypes.c_int),
        "spec_verify_rejection_ragged": ([P, ctypes.c_int, I64, I32, I64, I32, I32, P, P, P, I64, P, P, P, P, P,
                                          OUT, P, SZ, P], ctypes.c_int),
        "spec_verify_target_only_tree": ([P, ctypes.c_int, I64, I32, I32, I32, P, P, P, P, P, F, F, P, P, P, P,
                                          OUT, P, SZ, P], ctypes.c_int),
        "spec_verify_row_stats": ([P, ctypes.c_int, I64, I64, I32, P, P, P, P, P, P, P, P, SZ, P], ctypes.c_int),
        "spec_verify_set_stats_events": ([P, P], ctypes.c_int),
        "spec_verify_sparse_workspace_bytes": ([I64, I32, I32, I32, I32], SZ),
        "spec_verify_rejection_chain_sparse": ([P, ctypes.c_int, I64, I32, I32, I32, P, P, P, I32, I64, P, P, P, P, P,
                                                OUT, P, SZ, P], ctypes.c_int),
        "spec_verify_build_tree": ([P, P, I32, I32, P, P, P, P, P, P, P], ctypes.c_int),
        "spec_verify_sample_match_chain": ([P, ctypes.c_int, I64, I32, I32, I32, P, P, P, P, P, OUT, P, SZ, P],
                                           ctypes.c_int),
        "spec_verify_dspark_workspace_bytes": ([I32], SZ),
        "spec_verify_dspark_budget": ([P, I64, I32, P, I32, F, P], ctypes.c_int),
        "spec_verify_dspark_verify_lens": ([P, I32, I32, I64, I32, I32, I32, F, P, P, SZ, P], ctypes.c_int),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


# Argument checks.  The library takes raw device pointers and cannot tell a
# host pointer, a wrong element type or a short array from a good one, and the
# kernels would then read or write outside the arrays.  Every tensor is checked
# here before its pointer is passed: on the logits' device, of the element type
# the call reads, densely laid out (2-D arrays may have a row stride), and at
# least as large as the call reads.  None is passed on as NULL; whether an
# argument may be NULL is the library's decision (it returns SV_ERR_NULL_ARG).


def _require_cuda(t: torch.Tensor, name: str = "logits"):
    """The call's leading 2-D array: a CUDA tensor with dense rows; its device is the call's device."""
    if not isinstance(t, torch.Tensor) or t.dim() != 2:
        raise ValueError("%s must be a 2-D torch tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (got %s): the library has no CPU path" % (name, t.device))
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError("%s rows must be dense (stride 1 along a row)" % name)


def _arg(t: Optional[torch.Tensor], name: str, dtype: torch.dtype, numel: int, device) -> Optional[torch.Tensor]:
    """A 1-D (or dense N-D) array argument of at least numel elements."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % name)
    if t.device != device:
        raise ValueError("%s is on %s; the call runs on %s (the logits' device)" % (name, t.device, device))
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if t.numel() < numel:
        raise ValueError("%s has %d elements; the call reads %d" % (name, t.numel(), numel))
    return t


def _rows_arg(t: Optional[torch.Tensor], name: str, dtype: torch.dtype, rows: int, cols: int,
              device) -> Optional[torch.Tensor]:
    """A 2-D array argument [>= rows, >= cols] whose rows are dense (any row stride)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.dim() != 2:
        raise ValueError("%s must be a 2-D torch tensor" % name)
    if t.device != device:
        raise ValueError("%s is on %s; the call runs on %s (the logits' device)" % (name, t.device, device))
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if t.shape[0] < rows or t.shape[1] < cols:
        raise ValueError("%s is %s; the call reads [%d, %d]" % (name, tuple(t.shape), rows, cols))
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError("%s rows must be dense (stride 1 along a row)" % name)
    return t


def _check_out(out: "VerifyOutputs", batch: int, max_len: int, rows: int, device):
    i32, i64 = torch.int32, torch.int64
    _arg(out.accept_len, "out.accept_len", i32, batch, device)
    _arg(out.num_out, "out.num_out", i32, batch, device)
    _arg(out.out_tokens, "out.out_tokens", i32, batch * max_len, device)
    _arg(out.bonus, "out.bonus", i32, batch, device)
    _arg(out.accept_rows, "out.accept_rows", i32, batch * max_len, device)
    _arg(out.commit_cu, "out.commit_cu", i32, batch + 1, device)
    _arg(out.commit_src_slot, "out.commit_src_slot", i64, rows, device)
    _arg(out.commit_dst_pos, "out.commit_dst_pos", i64, rows, device)
    _arg(out.dev_status, "out.dev_status", i32, batch, device)


def _check_ws(ws: torch.Tensor, device):
    _arg(ws, "ws", torch.uint8, 0, device)


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype(logits: torch.Tensor) -> int:
    if logits.dtype == torch.bfloat16:
        return SV_BF16
    if logits.dtype == torch.float32:
        return SV_F32
    raise TypeError("logits must be bfloat16 or float32, got %s" % logits.dtype)


def _check(fn: str, code: int):
    if code != 0:
        lib = load_library()
        msg = lib.spec_verify_status_string(code).decode()
        if code == 7:
            msg += " (%s)" % lib.spec_verify_last_cuda_error().decode()
        raise SpecVerifyError(fn, code, msg)


def set_stats_events(start=None, stop=None):
    """Record torch CUDA events around the row-statistics kernel of later calls (None, None: stop).

    The events must already exist on the device (record them once first)."""
    h = lambda e: None if e is None else ctypes.c_void_p(e.cuda_event)
    _check("spec_verify_set_stats_events", load_library().spec_verify_set_stats_events(h(start), h(stop)))


def workspace_bytes(rows: int, batch: int, vocab: int, max_len: int) -> int:
    return int(load_library().spec_verify_workspace_bytes(rows, batch, vocab, max_len))


def workspace(rows: int, batch: int, vocab: int, max_len: int, device=None) -> torch.Tensor:
    """A zero-filled workspace (the library keeps its counters zero between calls)."""
    n = workspace_bytes(rows, batch, vocab, max_len)
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


@dataclass
class VerifyOutputs:
    accept_len: torch.Tensor
    num_out: torch.Tensor
    out_tokens: torch.Tensor
    bonus: torch.Tensor
    accept_rows: torch.Tensor
    commit_cu: torch.Tensor
    commit_src_slot: Optional[torch.Tensor]
    commit_dst_pos: Optional[torch.Tensor]
    dev_status: torch.Tensor  # int32 storage of uint32 bits

    @staticmethod
    def allocate(batch: int, max_len: int, rows: int, device=None, slots: bool = True) -> "VerifyOutputs":
        d = device or "cuda"
        i32 = dict(dtype=torch.int32, device=d)
        return VerifyOutputs(
            accept_len=torch.empty(batch, **i32), num_out=torch.empty(batch, **i32),
            out_tokens=torch.empty(batch, max_len, **i32), bonus=torch.empty(batch, **i32),
            accept_rows=torch.empty(batch, max_len, **i32), commit_cu=torch.empty(batch + 1, **i32),
            commit_src_slot=torch.full((max(rows, 1),), -1, dtype=torch.int64, device=d) if slots else None,
            commit_dst_pos=torch.full((max(rows, 1),), -1, dtype=torch.int64, device=d) if slots else None,
            dev_status=torch.empty(batch, **i32))

    def struct(self) -> SvOut:
        return SvOut(*[None if getattr(self, n) is None else getattr(self, n).data_ptr() for n, _ in SvOut._fields_])

    def to_numpy(self) -> dict:
        out = {}
        for n, _ in SvOut._fields_:
            t = getattr(self, n)
            if t is not None:
                a = t.cpu().numpy()
                out["status" if n == "dev_status" else n] = a.view("uint32") if n == "dev_status" else a
        return out


def _prep(out, ws, batch, max_len, rows, vocab, device, slots):
    if out is None:
        out = VerifyOutputs.allocate(batch, max_len, rows, device, slots)
    if ws is None:
        ws = workspace(rows, batch, vocab, max_len, device)
    _check_out(out, batch, max_len, rows, device)
    _check_ws(ws, device)
    return out, ws


def _chain_args(device, rows, batch, verify_ids, row_slots, seq_lens):
    _arg(verify_ids, "verify_ids", torch.int32, rows, device)
    _arg(row_slots, "row_slots", torch.int64, rows, device)
    _arg(seq_lens, "seq_lens", torch.int64, batch, device)


def greedy_chain(logits, verify_ids, m, *, row_slots=None, seq_lens=None, out=None, ws=None, stream=None):
    """Greedy chain verification of logits [batch*(m+1), V]."""
    lib = load_library()
    _require_cuda(logits)
    rows, V = logits.shape
    batch = rows // (m + 1)
    dev = logits.device
    _chain_args(dev, batch * (m + 1), batch, verify_ids, row_slots, seq_lens)
    out, ws = _prep(out, ws, batch, m + 1, rows, V, logits.device, row_slots is not None)
    st = out.struct()
    _check("spec_verify_greedy_chain", lib.spec_verify_greedy_chain(
        _ptr(logits), _dtype(logits), logits.stride(0), batch, m, V, _ptr(verify_ids), _ptr(row_slots),
        _ptr(seq_lens), ctypes.byref(st), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def rejection_chain(logits, verify_ids, m, q, temperature, u_accept, u_final, *, row_slots=None, seq_lens=None,
                    out=None, ws=None, stream=None):
    """p/q rejection chain verification of logits [batch*(m+1), V] with proposal rows q."""
    lib = load_library()
    _require_cuda(logits)
    rows, V = logits.shape
    batch = rows // (m + 1)
    dev, R = logits.device, batch * (m + 1)
    _chain_args(dev, R, batch, verify_ids, row_slots, seq_lens)
    _rows_arg(q, "q", torch.float32, R, V, dev)
    _arg(temperature, "temperature", torch.float32, batch, dev)
    _arg(u_accept, "u_accept", torch.float32, R, dev)
    _arg(u_final, "u_final", torch.float32, batch, dev)
    out, ws = _prep(out, ws, batch, m + 1, rows, V, logits.device, row_slots is not None)
    st = out.struct()
    _check("spec_verify_rejection_chain", lib.spec_verify_rejection_chain(
        _ptr(logits), _dtype(logits), logits.stride(0), batch, m, V, _ptr(verify_ids), _ptr(q), q.stride(0),
        _ptr(temperature), _ptr(u_accept), _ptr(u_final), _ptr(row_slots), _ptr(seq_lens), ctypes.byref(st),
        _ptr(ws), ws.numel(), _stream(stream)))
    return out


def sample_match_chain(logits, verify_ids, m, temperature, u_sample, *, row_slots=None, seq_lens=None, out=None,
                       ws=None, stream=None):
    """Verification by independent target sampling (u_sample per row) and prefix match."""
    lib = load_library()
    _require_cuda(logits)
    rows, V = logits.shape
    batch = rows // (m + 1)
    dev, R = logits.device, batch * (m + 1)
    _chain_args(dev, R, batch, verify_ids, row_slots, seq_lens)
    _arg(temperature, "temperature", torch.float32, batch, dev)
    _arg(u_sample, "u_sample", torch.float32, R, dev)
    out, ws = _prep(out, ws, batch, m + 1, rows, V, logits.device, row_slots is not None)
    st = out.struct()
    _check("spec_verify_sample_match_chain", lib.spec_verify_sample_match_chain(
        _ptr(logits), _dtype(logits), logits.stride(0), batch, m, V, _ptr(verify_ids), _ptr(temperature),
        _ptr(u_sample), _ptr(row_slots), _ptr(seq_lens), ctypes.byref(st), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def sparse_workspace(rows: int, batch: int, vocab: int, max_len: int, num_cands: int, device=None) -> torch.Tensor:
    lib = load_library()
    n = int(lib.spec_verify_sparse_workspace_bytes(rows, batch, vocab, max_len, num_cands))
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def rejection_chain_sparse(logits, verify_ids, m, cand_ids, cand_probs, temperature, u_accept, u_final, *,
                           row_slots=None, seq_lens=None, out=None, ws=None, stream=None):
    """p/q rejection chain whose q is given by candidate lists cand_ids / cand_probs [rows, K]."""
    lib = load_library()
    _require_cuda(logits)
    rows, V = logits.shape
    batch = rows // (m + 1)
    dev, R = logits.device, batch * (m + 1)
    _chain_args(dev, R, batch, verify_ids, row_slots, seq_lens)
    _rows_arg(cand_ids, "cand_ids", torch.int32, R, 0, dev)
    K = cand_ids.shape[1]
    _rows_arg(cand_probs, "cand_probs", torch.float32, R, K, dev)
    if cand_probs is not None and (cand_probs.shape[1] != K or (K > 1 and cand_probs.stride(0) != cand_ids.stride(0))):
        raise ValueError("cand_probs must have cand_ids' shape and row stride")
    _arg(temperature, "temperature", torch.float32, batch, dev)
    _arg(u_accept, "u_accept", torch.float32, R, dev)
    _arg(u_final, "u_final", torch.float32, batch, dev)
    if ws is None:
        ws = sparse_workspace(rows, batch, V, m + 1, K, logits.device)
    out, ws = _prep(out, ws, batch, m + 1, rows, V, logits.device, row_slots is not None)
    st = out.struct()
    _check("spec_verify_rejection_chain_sparse", lib.spec_verify_rejection_chain_sparse(
        _ptr(logits), _dtype(logits), logits.stride(0), batch, m, V, _ptr(verify_ids), _ptr(cand_ids),
        _ptr(cand_probs), K, cand_ids.stride(0), _ptr(temperature), _ptr(u_accept), _ptr(u_final),
        _ptr(row_slots), _ptr(seq_lens), ctypes.byref(st), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def rejection_ragged(logits, cu_seqlens, max_len, verify_ids, q, temperature, u_accept, u_final, *, row_slots=None,
                     seq_lens=None, out=None, ws=None, stream=None):
    """Ragged p/q rejection verification; cu_seqlens [B+1] int32 (lengths include the anchor)."""
    lib = load_library()
    _require_cuda(logits)
    rows, V = logits.shape
    dev = logits.device
    _arg(cu_seqlens, "cu_seqlens", torch.int32, 1, dev)
    batch = cu_seqlens.numel() - 1
    _chain_args(dev, rows, batch, verify_ids, row_slots, seq_lens)
    _rows_arg(q, "q", torch.float32, rows, V, dev)
    _arg(temperature, "temperature", torch.float32, batch, dev)
    _arg(u_accept, "u_accept", torch.float32, rows, dev)
    _arg(u_final, "u_final", torch.float32, batch, dev)
    out, ws = _prep(out, ws, batch, max_len, rows, V, logits.device, row_slots is not None)
    st = out.struct()
    _check("spec_verify_rejection_ragged", lib.spec_verify_rejection_ragged(
        _ptr(logits), _dtype(logits), logits.stride(0), batch, rows, max_len, V, _ptr(cu_seqlens), _ptr(verify_ids),
        _ptr(q), q.stride(0), _ptr(temperature), _ptr(u_accept), _ptr(u_final), _ptr(row_slots), _ptr(seq_lens),
        ctypes.byref(st), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def _tree_args(device, batch, nodes, tokens, parents, first_child, next_sibling, row_slots, seq_lens):
    n = batch * nodes
    _arg(tokens, "tokens", torch.int32, n, device)
    _arg(parents, "parents", torch.int32, n, device)
    _arg(first_child, "first_child", torch.int32, n, device)
    _arg(next_sibling, "next_sibling", torch.int32, n, device)
    _arg(row_slots, "row_slots", torch.int64, n, device)
    _arg(seq_lens, "seq_lens", torch.int64, batch, device)


def greedy_tree(logits, tokens, parents, *, first_child=None, next_sibling=None, row_slots=None, seq_lens=None,
                out=None, ws=None, stream=None):
    """Greedy tree verification; tokens / parents [batch, nodes], logits [batch*nodes, V]."""
    lib = load_library()
    _require_cuda(logits)
    rows, V = logits.shape
    batch, nodes = tokens.shape
    _tree_args(logits.device, batch, nodes, tokens, parents, first_child, next_sibling, row_slots, seq_lens)
    out, ws = _prep(out, ws, batch, nodes, rows, V, logits.device, row_slots is not None)
    st = out.struct()
    _check("spec_verify_greedy_tree", lib.spec_verify_greedy_tree(
        _ptr(logits), _dtype(logits), logits.stride(0), batch, nodes, V, _ptr(tokens), _ptr(parents),
        _ptr(first_child), _ptr(next_sibling), _ptr(row_slots), _ptr(seq_lens), ctypes.byref(st), _ptr(ws),
        ws.numel(), _stream(stream)))
    return out


def target_only_tree(logits, tokens, parents, temperature, u_accept, u_final, *, threshold_single=1.0,
                     threshold_acc=1.0, first_child=None, next_sibling=None, row_slots=None, seq_lens=None, out=None,
                     ws=None, stream=None):
    """Target-only tree sampling; u_accept [batch*nodes], u_final [batch]."""
    lib = load_library()
    _require_cuda(logits)
    rows, V = logits.shape
    batch, nodes = tokens.shape
    dev = logits.device
    _tree_args(dev, batch, nodes, tokens, parents, first_child, next_sibling, row_slots, seq_lens)
    _arg(temperature, "temperature", torch.float32, batch, dev)
    _arg(u_accept, "u_accept", torch.float32, batch * nodes, dev)
    _arg(u_final, "u_final", torch.float32, batch, dev)
    out, ws = _prep(out, ws, batch, nodes, rows, V, logits.device, row_slots is not None)
    st = out.struct()
    _check("spec_verify_target_only_tree", lib.spec_verify_target_only_tree(
        _ptr(logits), _dtype(logits), logits.stride(0), batch, nodes, V, _ptr(tokens), _ptr(parents),
        _ptr(first_child), _ptr(next_sibling), _ptr(temperature), float(threshold_single), float(threshold_acc),
        _ptr(u_accept), _ptr(u_final), _ptr(row_slots), _ptr(seq_lens), ctypes.byref(st), _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


def row_stats(logits, row_temp=None, probe=None, ws=None, stream=None) -> dict:
    """Row maximum, lowest argmax, Z (fp64), p at probe and flags for every row."""
    lib = load_library()
    _require_cuda(logits)
    rows, V = logits.shape
    d = logits.device
    _arg(row_temp, "row_temp", torch.float32, rows, d)
    _arg(probe, "probe", torch.int32, rows, d)
    res = {"max": torch.empty(rows, dtype=torch.float32, device=d),
           "argmax": torch.empty(rows, dtype=torch.int32, device=d),
           "z": torch.empty(rows, dtype=torch.float64, device=d),
           "p": torch.empty(rows, dtype=torch.float32, device=d) if probe is not None else None,
           "flags": torch.empty(rows, dtype=torch.int32, device=d)}
    if ws is None:
        ws = workspace(rows, 1, V, 1, d)
    _check_ws(ws, d)
    _check("spec_verify_row_stats", lib.spec_verify_row_stats(
        _ptr(logits), _dtype(logits), logits.stride(0), rows, V, _ptr(row_temp), _ptr(probe), _ptr(res["max"]),
        _ptr(res["argmax"]), _ptr(res["z"]), _ptr(res["p"]), _ptr(res["flags"]), _ptr(ws), ws.numel(),
        _stream(stream)))
    return res


def dspark_budget(hist_survival, num_requests: int, sps, eps: float = 0.0) -> int:
    """Host budget K* from historical survival scores and a speed table indexed by target rows."""
    lib = load_library()
    h = np.ascontiguousarray(np.asarray(hist_survival, dtype=np.float32).ravel())
    t = np.ascontiguousarray(np.asarray(sps, dtype=np.float32).ravel())
    k = ctypes.c_int32(-1)
    _check("spec_verify_dspark_budget", lib.spec_verify_dspark_budget(
        ctypes.c_void_p(h.ctypes.data) if h.size else None, h.size, int(num_requests),
        ctypes.c_void_p(t.ctypes.data) if t.size else None, t.size, float(eps), ctypes.byref(k)))
    return int(k.value)


def dspark_workspace(num_requests: int, device=None) -> torch.Tensor:
    lib = load_library()
    return torch.zeros(int(lib.spec_verify_dspark_workspace_bytes(int(num_requests))), dtype=torch.uint8,
                       device=device)


def dspark_verify_lens(survival, budget: int, *, min_len: int = 1, max_len: Optional[int] = None, eps: float = 0.0,
                       out=None, ws=None, stream=None) -> torch.Tensor:
    """verify_lens [R] (int32, on survival's device) from the current survival [R, D]."""
    lib = load_library()
    _require_cuda(survival, "survival")
    R, D = survival.shape
    dev = survival.device
    _rows_arg(survival, "survival", torch.float32, R, D, dev)
    if max_len is None:
        max_len = D + 1
    if out is None:
        out = torch.empty(R, dtype=torch.int32, device=survival.device)
    if ws is None:
        ws = dspark_workspace(R, survival.device)
    _arg(out, "out", torch.int32, R, dev)
    _check_ws(ws, dev)
    _check("spec_verify_dspark_verify_lens", lib.spec_verify_dspark_verify_lens(
        _ptr(survival), R, D, survival.stride(0), int(budget), int(min_len), int(max_len), float(eps), _ptr(out),
        _ptr(ws), ws.numel(), _stream(stream)))
    return out


def build_tree(parents, seq_lens=None, stream=None, out: Optional[dict] = None) -> dict:
    """Positions, ancestor mask, retrieve index and child / sibling links from parents [B, N] (int32, device).

    out: optional preallocated results with the keys and shapes this function returns."""
    lib = load_library()
    _require_cuda(parents, "parents")
    B, N = parents.shape
    d = parents.device
    _arg(parents, "parents", torch.int32, B * N, d)
    _arg(seq_lens, "seq_lens", torch.int64, B, d)
    res = out if out is not None else {
        "positions": torch.empty(B, N, dtype=torch.int64, device=d),
        "mask": torch.empty(B, N, N, dtype=torch.uint8, device=d),
        "retrieve_index": torch.empty(B, N, dtype=torch.int32, device=d),
        "first_child": torch.empty(B, N, dtype=torch.int32, device=d),
        "next_sibling": torch.empty(B, N, dtype=torch.int32, device=d),
        "status": torch.empty(B, dtype=torch.int32, device=d)}
    for k, dt, n in (("positions", torch.int64, B * N), ("mask", torch.uint8, B * N * N),
                     ("retrieve_index", torch.int32, B * N), ("first_child", torch.int32, B * N),
                     ("next_sibling", torch.int32, B * N), ("status", torch.int32, B)):
        if res.get(k) is None:
            raise ValueError("build_tree: out lacks %r" % k)
        _arg(res[k], "out[%r]" % k, dt, n, d)
    _check("spec_verify_build_tree", lib.spec_verify_build_tree(
        _ptr(parents), _ptr(seq_lens), B, N, _ptr(res["positions"]), _ptr(res["mask"]), _ptr(res["retrieve_index"]),
        _ptr(res["first_child"]), _ptr(res["next_sibling"]), _ptr(res["status"]), _stream(stream)))
    return res
