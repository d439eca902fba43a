"""Sparse-q rejection (candidate lists) on the GPU vs the oracle over the scattered q.

Same bar as the dense chain: token decisions, lengths, commit lists and status
bits bit-exact on every request whose decisions are not within 1e-6 of a
threshold (counted and reported).
"""
import dataclasses

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from reject_row_vocab_gb300 import _build  # noqa: E402

_build.build()
from reject_row_vocab_gb300 import device_workload as dw  # noqa: E402
from reject_row_vocab_gb300 import workload as wl  # noqa: E402
from tests.gpu_compare import compare, oracle_outputs  # noqa: E402


def run_gpu(w, ws=None):
    d = dw.DeviceInputs.from_workload(w)
    o = dw.run(w, d, ws=dw.workspace_for(w) if ws is None else ws)
    torch.cuda.synchronize()
    return o.to_numpy()


def check(w):
    g = run_gpu(w)
    o = oracle_outputs(w)
    r = compare(w, g, o)
    print(w.name, r)
    return g, o


@pytest.mark.parametrize("batch,m,vocab,K,dtype,pad,T", [
    (4, 3, 300, 8, "f32", 0, 0.9),
    (6, 5, 2053, 16, "bf16", 2, 0.8),      # ragged last tile
    (8, 7, 20011, 16, "bf16", 0, 1.0),
    (5, 4, 4099, 1, "f32", 0, 0.7),        # one-hot q: alpha = p(d)
    (3, 6, 300, 300, "bf16", 0, 1.2),      # every id a candidate
    (7, 2, 65536, 64, "bf16", 5, 0.6),
])
def test_sparse_chain_matches_oracle(batch, m, vocab, K, dtype, pad, T):
    w = wl.rejection_chain_sparse(batch=batch, m=m, vocab=vocab, K=K, dtype=dtype, pad=pad, temperature=T,
                                  boost=2.0, seed=batch * 1000 + vocab + K)
    check(w)


def test_sparse_degenerate_inputs():
    w = wl.rejection_chain_sparse(batch=9, m=4, vocab=1000, K=6, pad=2, seed=77)
    ids, pr, T = w.cand_ids.copy(), w.cand_probs.copy(), w.temperature.copy()
    L = w.max_len
    ids[1 * L + 2, 3] = 1000            # out of range in a tested row: flagged
    ids[2 * L + L - 1, 0] = -7          # last row of request 2: never tested, not flagged
    ids[3 * L, 1] = ids[3 * L, 0]       # repeated id: probabilities add up
    T[4] = 0.0                          # greedy request among sampling ones
    T[5] = float("nan")                 # greedy too
    pr[6 * L:7 * L] *= 0.5              # q need not sum to 1
    # request 7 rejects its first draft (q(d) huge) and its residual row lists ids past V and below -1 with
    # negative probabilities: both are ignored, so no weight appears outside the vocabulary
    r = 7 * L
    d = w.verify_ids[r + 1]
    pr[r, ids[r] == d] = 1e6
    ids[r, 6], pr[r, 6] = w.vocab + 5, -1.0  # inside the last (ragged) tile
    ids[r, 7], pr[r, 7] = -3, -1.0
    w2 = dataclasses.replace(w, cand_ids=ids, cand_probs=pr, temperature=T)
    g, o = check(w2)
    assert (int(g["status"][1]) & 1) == 1 and (int(g["status"][2]) & 1) == 0
    assert int(o["accept_len"][7]) == 0 and (int(g["status"][7]) & 1) == 1
    assert 0 <= int(g["bonus"][7]) < w.vocab


def test_full_size_sparse_dflash_block():
    """The DFlash block shape (64 requests x 16 rows, V = 151936, bf16) with K = 16 candidates per row."""
    w = wl.rejection_chain_sparse(batch=64, m=15, vocab=151936, K=16, dtype="bf16", boost=0.0, temperature=1.0,
                                  noise_sigma=1.5, sigma=3.0, seed=1004)
    g, o = check(w)
    # residual draws may leave the candidate set: the proposal does not confine the output
    L = w.max_len
    outside = 0
    for b in range(w.batch):
        s = int(o["accept_len"][b])
        if s < L - 1:
            if int(g["bonus"][b]) not in set(w.cand_ids[b * L + s].tolist()):
                outside += 1
    print("residual tokens outside the candidate list:", outside)


def test_sparse_workspace_reuse_and_validation():
    w = wl.rejection_chain_sparse(batch=5, m=3, vocab=5000, K=8, seed=12)
    ws = dw.workspace_for(w)
    a = run_gpu(w, ws=ws)
    b = run_gpu(w, ws=ws)
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    from reject_row_vocab_gb300 import specverify as sv
    d = dw.DeviceInputs.from_workload(w)
    with pytest.raises(sv.SpecVerifyError):  # num_cands > ldc
        lib = sv.load_library()
        out = dw.outputs_for(w)
        st = out.struct()
        import ctypes
        sv._check("spec_verify_rejection_chain_sparse", lib.spec_verify_rejection_chain_sparse(
            sv._ptr(d["logits"]), sv._dtype(d["logits"]), d["logits"].stride(0), w.batch, w.m, w.vocab,
            sv._ptr(d["verify_ids"]), sv._ptr(d["cand_ids"]), sv._ptr(d["cand_probs"]), 9, 8,
            sv._ptr(d["temperature"]), sv._ptr(d["u_accept"]), sv._ptr(d["u_final"]), sv._ptr(d["row_slots"]),
            sv._ptr(d["seq_lens"]), ctypes.byref(st), sv._ptr(ws), ws.numel(), None))
