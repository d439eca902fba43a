"""The no-allocation rejection entry point gives the same results as the workspace one.

spec_verify_rejection_chain_noalloc serves callers that cannot hand the library
any device scratch memory (a plugin given only its input and output buffers, an
engine that has already reserved all device memory): it runs the same kernels
on a fixed scratch area inside the library.  This file is collected last so a
stop-at-first-failure run has already run every other test; it also passes on
its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from reject_row_vocab_gb300 import _build  # noqa: E402

_build.build()
from reject_row_vocab_gb300 import device_workload as dw  # noqa: E402
from reject_row_vocab_gb300 import specverify as sv  # noqa: E402
from reject_row_vocab_gb300 import workload as wl  # noqa: E402
from tests.gpu_compare import compare, oracle_outputs  # noqa: E402


def _entry():
    lib = sv.load_library()
    fn = lib.spec_verify_rejection_chain_noalloc
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    fn.argtypes = [P, ctypes.c_int, I64, I32, I32, I32, P, P, I64, P, P, P, P, P, ctypes.POINTER(sv.SvOut), P]
    fn.restype = ctypes.c_int
    return fn


def _call_noalloc(fn, w, d, out, batch=None, vocab=None):
    logits = d["logits"]
    st = out.struct()
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return fn(p(logits), sv._dtype(logits), logits.stride(0), w.batch if batch is None else batch, w.max_len - 1,
              w.vocab if vocab is None else vocab, p(d["verify_ids"]), p(d["q"]), d["q"].stride(0),
              p(d["temperature"]), p(d["u_accept"]), p(d["u_final"]), p(d["row_slots"]), p(d["seq_lens"]),
              ctypes.byref(st), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_no_alloc_entry_matches_workspace_entry_on_two_calls():
    fn = _entry()
    cases = [wl.rejection_chain(batch=12, m=7, vocab=20011, dtype="bf16", boost=2.0, seed=77, name="noalloc_a"),
             wl.rejection_chain(batch=5, m=3, vocab=4099, dtype="f32", temperature=0.7, seed=78, name="noalloc_b")]
    for w in cases:  # two calls in a row, different sizes: the shared area's leftovers must not matter
        d = dw.DeviceInputs.from_workload(w)
        ref = dw.run(w, d).to_numpy()  # the regular entry point with its own workspace
        out = dw.outputs_for(w)
        assert _call_noalloc(fn, w, d, out) == 0
        torch.cuda.synchronize()
        got = out.to_numpy()
        for k, v in ref.items():
            assert np.array_equal(got[k], v), (w.name, k)
        compare(w, got, oracle_outputs(w))


def test_no_alloc_entry_clears_what_an_earlier_call_left():
    """Each call clears the shared area's counter words itself: dirty counters (set on purpose, or left by a
    call whose waits ran out) do not change the next call's results."""
    fn = _entry()
    lib = sv.load_library()
    lib.spec_verify_noalloc_fill_counters.argtypes = [ctypes.c_uint32, ctypes.c_void_p]
    lib.spec_verify_set_hand_off_limit_ns.argtypes = [ctypes.c_uint64]
    w = wl.rejection_chain(batch=12, m=7, vocab=20011, dtype="bf16", boost=2.0, seed=80, name="noalloc_dirty")
    d = dw.DeviceInputs.from_workload(w)
    want = oracle_outputs(w)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for value in (0xFF, 0x01):
        assert lib.spec_verify_noalloc_fill_counters(value, stream) == 0
        out = dw.outputs_for(w)
        assert _call_noalloc(fn, w, d, out) == 0
        torch.cuda.synchronize()
        compare(w, out.to_numpy(), want)
    assert lib.spec_verify_set_hand_off_limit_ns(2000) == 0
    try:
        out = dw.outputs_for(w)
        assert _call_noalloc(fn, w, d, out) == 0
        torch.cuda.synchronize()
    finally:
        lib.spec_verify_set_hand_off_limit_ns(0)
    assert np.all(out.to_numpy()["status"] & 64)  # SV_DEV_TIMEOUT
    out = dw.outputs_for(w)
    assert _call_noalloc(fn, w, d, out) == 0
    torch.cuda.synchronize()
    compare(w, out.to_numpy(), want)


def test_no_alloc_entry_rejects_sizes_beyond_its_scratch():
    fn = _entry()
    w = wl.rejection_chain(batch=2, m=3, vocab=256, dtype="bf16", seed=79)
    d = dw.DeviceInputs.from_workload(w)
    out = dw.outputs_for(w)
    need = sv.workspace_bytes(4096 * 16, 4096, 1 << 20, 16)
    assert need > (4 << 20)
    # the size check happens before anything is read or enqueued
    assert _call_noalloc(fn, w, d, out, batch=4096, vocab=1 << 20) == 6  # SV_ERR_WORKSPACE_TOO_SMALL
    # so do the argument checks: nothing of a refused call reaches the stream
    out.commit_cu.fill_(-5)
    st = out.struct()
    null = None
    assert fn(ctypes.c_void_p(d["logits"].data_ptr()), sv._dtype(d["logits"]), d["logits"].stride(0), w.batch,
              w.max_len - 1, w.vocab, null, ctypes.c_void_p(d["q"].data_ptr()), d["q"].stride(0),
              ctypes.c_void_p(d["temperature"].data_ptr()), ctypes.c_void_p(d["u_accept"].data_ptr()),
              ctypes.c_void_p(d["u_final"].data_ptr()), null, null, ctypes.byref(st),
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 1  # SV_ERR_NULL_ARG
    torch.cuda.synchronize()
    assert np.all(out.commit_cu.cpu().numpy() == -5)
