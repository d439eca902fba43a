"""A fixed-length p/q rejection chain and the same batch given as a ragged block.

A chain of B requests with L rows each, and the ragged block with
cu_seqlens = b * L over the same arrays, describe the same verification: the
streaming pass maps rows to requests differently (a fixed stride against a
search of the offsets) but merges every row in the same chunk order, and the
acceptance and sampling read the same rows, so the outputs must agree bit
for bit, and both must match the oracle under the parity rule.  The shapes
span one tile per row, a ragged last tile, 32 and 33 rows per request, bonus
rows only, greedy requests inside a sampling batch, and repeated calls on one
workspace (the call's counters rewind themselves).
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

KEYS = ("accept_len", "num_out", "out_tokens", "bonus", "accept_rows", "commit_cu", "status")


def _ragged_run(w, d):
    L = w.max_len
    cu = torch.arange(0, (w.batch + 1) * L, L, dtype=torch.int32, device="cuda")
    ws = sv.workspace(w.rows, w.batch, w.vocab, L)
    o = sv.rejection_ragged(d["logits"], cu, L, d["verify_ids"], d["q"], d["temperature"], d["u_accept"],
                            d["u_final"], row_slots=d["row_slots"], seq_lens=d["seq_lens"], ws=ws)
    torch.cuda.synchronize()
    return o.to_numpy()


def _same(a, b):
    for k in KEYS:
        assert np.array_equal(a[k], b[k]), k
    for k in ("commit_src_slot", "commit_dst_pos"):
        if a.get(k) is not None:
            n = int(a["commit_cu"][-1])
            assert np.array_equal(a[k][:n], b[k][:n]), k


@pytest.mark.parametrize("batch,m,vocab,dtype,seed", [
    (8, 7, 151936, "bf16", 501),     # the 8 x 8 chain
    (64, 15, 151936, "bf16", 502),   # the DFlash block shape
    (3, 0, 1000, "f32", 503),        # bonus rows only
    (5, 31, 4099, "bf16", 504),      # 32 rows per request, ragged last tile
    (40, 3, 32000, "f32", 505),
    (1, 4, 7, "bf16", 506),          # one tile per row
    (200, 3, 256, "f32", 507),       # many requests per sampler block
    (4, 32, 5000, "bf16", 508),      # 33 rows per request
])
def test_fixed_chain_matches_ragged_block_and_oracle(batch, m, vocab, dtype, seed):
    w = wl.rejection_chain(batch=batch, m=m, vocab=vocab, dtype=dtype, seed=seed, name="fixed_vs_ragged")
    d = dw.DeviceInputs.from_workload(w)
    ws = dw.workspace_for(w)
    out = dw.outputs_for(w)
    g = dw.run(w, d, out=out, ws=ws).to_numpy()
    torch.cuda.synchronize()
    _same(g, _ragged_run(w, d))
    compare(w, g, oracle_outputs(w))
    # the call's counters rewind themselves: the same workspace gives the same outputs again
    g2 = dw.run(w, d, out=out, ws=ws).to_numpy()
    torch.cuda.synchronize()
    _same(g, g2)


def test_fixed_chain_greedy_requests_inside_a_sampling_batch():
    # temperature 0 for some requests: greedy acceptance and no draw for those
    w = wl.rejection_chain(batch=24, m=5, vocab=50000, dtype="bf16", seed=509, name="fixed_vs_ragged_mixed_T")
    w.temperature[::3] = 0.0
    d = dw.DeviceInputs.from_workload(w)
    g = dw.run(w, d, ws=dw.workspace_for(w)).to_numpy()
    torch.cuda.synchronize()
    _same(g, _ragged_run(w, d))
    compare(w, g, oracle_outputs(w))
