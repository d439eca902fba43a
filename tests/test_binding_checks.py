"""Argument checks of the Python binding (no GPU).

The library takes raw device pointers, so the binding checks every tensor's
device, element type, layout and size before passing its pointer.  These
tests run the binding on CPU tensors with the library's verification entry
points replaced by stubs (and the CUDA requirement on the logits lifted), so
that the checks themselves can be exercised here: every workload shape the
GPU tests use must pass them, and each kind of bad argument must be refused
before the library is called.
"""
import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from reject_row_vocab_gb300 import device_workload as dw  # noqa: E402
from reject_row_vocab_gb300 import specverify as sv  # noqa: E402
from reject_row_vocab_gb300 import workload as wl  # noqa: E402

ENTRY = ("spec_verify_greedy_chain", "spec_verify_greedy_tree", "spec_verify_rejection_chain",
         "spec_verify_rejection_ragged", "spec_verify_target_only_tree", "spec_verify_sample_match_chain",
         "spec_verify_rejection_chain_sparse", "spec_verify_row_stats", "spec_verify_dspark_verify_lens",
         "spec_verify_build_tree")


class _StubLib:
    """The real library for sizes and strings; verification entry points only record their calls."""

    def __init__(self, real):
        self.real, self.calls = real, []

    def __getattr__(self, name):
        if name in ENTRY:
            return lambda *a: self.calls.append(name) or 0
        return getattr(self.real, name)


@pytest.fixture
def cpu_binding(monkeypatch):
    from reject_row_vocab_gb300 import _build
    _build.build()
    stub = _StubLib(sv.load_library())
    monkeypatch.setattr(sv, "load_library", lambda: stub)
    monkeypatch.setattr(sv, "_stream", lambda s: None)
    monkeypatch.setattr(sv, "_require_cuda", lambda t, name="logits": None)
    return stub


def _workloads():
    # the five workload layouts at a small vocabulary (the checks are relative to the shapes)
    yield wl.config(1)
    yield wl.config(2, vocab=2048)
    yield wl.config(3, mode="greedy_tree", vocab=2048)
    yield wl.config(3, mode="target_only_tree", vocab=2048)
    yield wl.config(4, vocab=1024)
    yield wl.config(5, vocab=1024)
    yield wl.rejection_chain(batch=3, m=4, vocab=1001, dtype="f32", seed=3)
    yield wl.rejection_chain(batch=17, m=0, vocab=3001, dtype="bf16", seed=8)
    yield wl.rejection_chain_sparse(batch=4, m=3, vocab=1000, dtype="bf16", K=8, sigma=3.0, boost=0.0,
                                    temperature=1.0, noise_sigma=1.0, pad=0, seed=1, name="sparse")
    import dataclasses
    w = wl.config(2, vocab=2048)
    yield dataclasses.replace(w, kind="sample_match_chain", q=None, name="match")


def test_every_workload_passes_the_checks(cpu_binding):
    for w in _workloads():
        d = dw.DeviceInputs.from_workload(w, device="cpu")
        out = dw.outputs_for(w, device="cpu")
        ws = dw.workspace_for(w, device="cpu")
        dw.run(w, d, out=out, ws=ws)
        if w.kind in ("greedy_tree", "target_only_tree") and w.first_child is not None:
            dw.run(w, d, out=out, ws=ws, use_lists=True)
    assert len(cpu_binding.calls) >= 9


def test_direct_calls_pass_the_checks(cpu_binding):
    rows, V = 7, 1000
    t = dw.padded_rows(torch.zeros((rows, V), dtype=torch.bfloat16), "cpu")
    sv.row_stats(t, row_temp=torch.ones(rows), probe=torch.zeros(rows, dtype=torch.int32),
                 ws=torch.zeros(sv.workspace_bytes(rows, 1, V, 1), dtype=torch.uint8))
    sv.greedy_chain(torch.zeros((0, 64), dtype=torch.bfloat16), torch.zeros(0, dtype=torch.int32), 3,
                    ws=torch.zeros(sv.workspace_bytes(0, 0, 64, 4), dtype=torch.uint8),
                    out=sv.VerifyOutputs.allocate(0, 4, 0, "cpu", slots=False))
    surv = torch.rand((40, 8))[:, :6]  # a row-strided view, as the scheduler test passes
    sv.dspark_verify_lens(surv, 50, ws=torch.zeros(64 << 10, dtype=torch.uint8))
    par = torch.tensor([[-1, 0, 0, 1]], dtype=torch.int32)
    res = sv.build_tree(par, torch.tensor([7]))
    sv.build_tree(par, None, out=res)  # preallocated results pass the same checks
    bad = dict(res, mask=res["mask"].int())
    with pytest.raises(TypeError):
        sv.build_tree(par, None, out=bad)
    with pytest.raises(TypeError):
        sv.build_tree(torch.tensor([[-1, 0, 0, 1]]), None)  # int64 parents
    with pytest.raises(TypeError):
        sv.dspark_verify_lens(surv.double(), 50)
    assert cpu_binding.calls == ["spec_verify_row_stats", "spec_verify_greedy_chain", "spec_verify_dspark_verify_lens",
                                 "spec_verify_build_tree", "spec_verify_build_tree"]


def _chain_case():
    w = wl.rejection_chain(batch=3, m=4, vocab=1001, dtype="bf16", seed=3)
    d = dw.DeviceInputs.from_workload(w, device="cpu")
    return w, d, dict(out=dw.outputs_for(w, device="cpu"), ws=dw.workspace_for(w, device="cpu"))


@pytest.mark.parametrize("bad", ["short_u", "ids_int64", "q_f64", "q_short_rows", "noncontig_ids",
                                 "temperature_f64", "out_short", "ws_f32", "q_col_strided"])
def test_bad_arguments_are_refused_before_the_library(cpu_binding, bad):
    w, d, kw = _chain_case()
    args = dict(verify_ids=d["verify_ids"], q=d["q"], temperature=d["temperature"], u_accept=d["u_accept"],
                u_final=d["u_final"])
    if bad == "short_u":
        args["u_accept"] = args["u_accept"][:-1]
    elif bad == "ids_int64":
        args["verify_ids"] = args["verify_ids"].long()
    elif bad == "q_f64":
        args["q"] = args["q"].double()
    elif bad == "q_short_rows":
        args["q"] = args["q"][:-1]
    elif bad == "noncontig_ids":
        args["verify_ids"] = torch.stack([args["verify_ids"], args["verify_ids"]], 1)[:, 0]
    elif bad == "temperature_f64":
        args["temperature"] = args["temperature"].double()
    elif bad == "out_short":
        kw["out"] = sv.VerifyOutputs.allocate(w.batch - 1, w.max_len, w.rows, "cpu", slots=False)
    elif bad == "ws_f32":
        kw["ws"] = kw["ws"].float()
    elif bad == "q_col_strided":
        args["q"] = torch.zeros((w.rows, 2 * w.vocab))[:, ::2]
    with pytest.raises((TypeError, ValueError)):
        sv.rejection_chain(d["logits"], args["verify_ids"], w.max_len - 1, args["q"], args["temperature"],
                           args["u_accept"], args["u_final"], **kw)
    assert cpu_binding.calls == []


def test_cpu_logits_fail_loudly_without_a_gpu():
    from reject_row_vocab_gb300 import _build
    _build.build()
    w = wl.rejection_chain(batch=2, m=2, vocab=100, dtype="f32", seed=1)
    d = dw.DeviceInputs.from_workload(w, device="cpu")
    with pytest.raises(ValueError, match="CUDA"):
        dw.run(w, d, out=dw.outputs_for(w, device="cpu"), ws=dw.workspace_for(w, device="cpu"))


def test_tensor_on_another_device_is_refused():
    t = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(ValueError, match="device"):
        sv._arg(t, "x", torch.int32, 4, torch.device("meta"))
    assert sv._arg(None, "x", torch.int32, 4, torch.device("cpu")) is None
    assert sv._arg(t, "x", torch.int32, 4, t.device) is t
    with pytest.raises(ValueError):
        sv._arg(t, "x", torch.int32, 5, t.device)
    np.testing.assert_equal(sv._rows_arg(torch.zeros((3, 8))[:, :5], "y", torch.float32, 3, 5,
                                         torch.device("cpu")).shape, (3, 5))
