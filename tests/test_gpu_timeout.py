"""The statistics kernel's bounded waits, made to run out on purpose.

Every wait inside the row-statistics kernel is bounded; when one gives up, the
kernel stops, waits (with the normal limit) for its own bulk copies still in
flight, and raises the workspace error word, and the call's requests report
SV_DEV_TIMEOUT.  spec_verify_set_hand_off_limit_ns puts the kernel into its
expiry test: the in-CTA hand-off waits get a short limit and one wait is on a
barrier that nothing completes, so the path runs for certain — with no GPU
fault, no stalled copy engine, and the context still usable afterwards.
"""
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

SV_DEV_TIMEOUT = 64


def _expired_call(w, d, ws, limit_ns):
    lib = sv.load_library()
    lib.spec_verify_set_hand_off_limit_ns.argtypes = [__import__("ctypes").c_uint64]
    assert lib.spec_verify_set_hand_off_limit_ns(limit_ns) == 0
    try:
        res = dw.run(w, d, ws=ws)
        torch.cuda.synchronize()
    finally:
        lib.spec_verify_set_hand_off_limit_ns(0)
    return res.to_numpy()


@pytest.mark.parametrize("kind", ["rejection_chain", "greedy_tree", "ragged"])
def test_expired_waits_report_timeout_and_the_next_call_is_exact(kind):
    if kind == "rejection_chain":
        w = wl.rejection_chain(batch=16, m=7, vocab=151936, dtype="bf16", seed=91, name="expiry_chain")
    elif kind == "greedy_tree":
        w = wl.eagle2_tree(batch=4, topk=3, depth=3, keep=8, vocab=32000, mode="greedy_tree", seed=92,
                           name="expiry_tree")
    else:
        w = wl.ragged_block(batch=48, max_len=8, vocab=50000, seed=93, name="expiry_ragged")
    d = dw.DeviceInputs.from_workload(w)
    ws = dw.workspace_for(w)
    for limit in (2000, 1):  # a few microseconds, and effectively none
        g = _expired_call(w, d, ws, limit)
        assert np.all(g["status"] & SV_DEV_TIMEOUT), g["status"]
        assert g["commit_cu"][0] == 0 and np.all(np.diff(g["commit_cu"]) == g["num_out"])
        ws.zero_()  # the documented recovery: zero-fill the workspace once
        g = dw.run(w, d, ws=ws).to_numpy()
        torch.cuda.synchronize()
        assert not np.any(g["status"] & SV_DEV_TIMEOUT)
        compare(w, g, oracle_outputs(w))
