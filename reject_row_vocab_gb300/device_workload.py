"""Move a synthetic workload to the GPU and dispatch it to the matching entry point.

Marshalling only: the verification itself runs in libspecverify.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

from . import specverify as sv
from .workload import Workload

_ARRAYS = ("cu_seqlens", "verify_ids", "q", "cand_ids", "cand_probs", "temperature", "u_accept", "u_final",
           "tokens", "parents", "first_child", "next_sibling", "row_slots", "seq_lens")


def padded_rows(t: torch.Tensor, device) -> torch.Tensor:
    """A [rows, V] device view whose row stride is a multiple of 16 bytes (the library's layout rule)."""
    rows, V = t.shape
    per = 16 // t.element_size()
    ld = (V + per - 1) // per * per
    if ld == V:
        return t.to(device)
    buf = torch.zeros((rows, ld), dtype=t.dtype, device=device)
    view = buf[:, :V]
    view.copy_(t)
    return view


def _to_tensor(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    if a.dtype == np.uint32:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int32))
    return torch.from_numpy(np.ascontiguousarray(a))


@dataclass
class DeviceInputs:
    """Device copies of every input array of a workload (logits as bf16 or fp32)."""
    t: dict = field(default_factory=dict)

    @staticmethod
    def from_workload(w: Workload, device="cuda", pin: bool = False) -> "DeviceInputs":
        d = DeviceInputs()
        d.t["logits"] = _to_tensor(w.logits)
        for k in _ARRAYS:
            v = getattr(w, k)
            if v is not None:
                d.t[k] = _to_tensor(v)
        for k, v in d.t.items():
            if pin:
                d.t[k] = v.pin_memory()
            elif k in ("logits", "q"):
                d.t[k] = padded_rows(v, device)
            else:
                d.t[k] = v.to(device)
        return d

    def __getitem__(self, k):
        return self.t.get(k)

    def nbytes(self) -> int:
        return sum(v.numel() * v.element_size() for v in self.t.values())

    def copy_from(self, host: "DeviceInputs", non_blocking: bool = True) -> int:
        """Copy every array from (pinned) host tensors into these device tensors; returns bytes."""
        n = 0
        for k, v in host.t.items():
            self.t[k].copy_(v, non_blocking=non_blocking)
            n += v.numel() * v.element_size()
        return n


def kind_max_len(w: Workload) -> int:
    return w.nodes if w.nodes else w.max_len


def run(w: Workload, d: DeviceInputs, out: Optional[sv.VerifyOutputs] = None, ws: Optional[torch.Tensor] = None,
        stream=None, use_lists: bool = False) -> sv.VerifyOutputs:
    """Verify the workload on the GPU through the entry point its kind names."""
    kw = dict(row_slots=d["row_slots"], seq_lens=d["seq_lens"], out=out, ws=ws, stream=stream)
    if w.kind == "greedy_chain":
        return sv.greedy_chain(d["logits"], d["verify_ids"], w.max_len - 1, **kw)
    if w.kind == "rejection_chain":
        return sv.rejection_chain(d["logits"], d["verify_ids"], w.max_len - 1, d["q"], d["temperature"],
                                  d["u_accept"], d["u_final"], **kw)
    if w.kind == "sample_match_chain":
        return sv.sample_match_chain(d["logits"], d["verify_ids"], w.max_len - 1, d["temperature"], d["u_accept"], **kw)
    if w.kind == "rejection_chain_sparse":
        return sv.rejection_chain_sparse(d["logits"], d["verify_ids"], w.max_len - 1, d["cand_ids"], d["cand_probs"],
                                         d["temperature"], d["u_accept"], d["u_final"], **kw)
    if w.kind == "rejection_ragged":
        return sv.rejection_ragged(d["logits"], d["cu_seqlens"], w.max_len, d["verify_ids"], d["q"],
                                   d["temperature"], d["u_accept"], d["u_final"], **kw)
    lists = dict(first_child=d["first_child"], next_sibling=d["next_sibling"]) if use_lists else {}
    if w.kind == "greedy_tree":
        return sv.greedy_tree(d["logits"], d["tokens"], d["parents"], **lists, **kw)
    if w.kind == "target_only_tree":
        return sv.target_only_tree(d["logits"], d["tokens"], d["parents"], d["temperature"], d["u_accept"],
                                   d["u_final"], threshold_single=w.threshold_single,
                                   threshold_acc=w.threshold_acc, **lists, **kw)
    raise ValueError(w.kind)


def workspace_for(w: Workload, device="cuda") -> torch.Tensor:
    if w.cand_ids is not None:
        return sv.sparse_workspace(w.rows, w.batch, w.vocab, kind_max_len(w), w.cand_ids.shape[1], device)
    return sv.workspace(w.rows, w.batch, w.vocab, kind_max_len(w), device)


def outputs_for(w: Workload, device="cuda") -> sv.VerifyOutputs:
    return sv.VerifyOutputs.allocate(w.batch, kind_max_len(w), w.rows, device, slots=w.row_slots is not None)
