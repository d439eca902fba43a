"""Pins of the sparse-q (candidate list) oracle, no GPU.

[E2D] §6.5: the selector's q has K nonzeros given by candidate ids; it is
scattered into vocabulary coordinates before rejection, and tokens outside
the candidates can still come out through the residual.
"""
import dataclasses

import numpy as np

import oracle
from reject_row_vocab_gb300 import workload as wl


def test_scatter_by_hand():
    q, bad = oracle.scatter_candidates([[3, -1, 3, 1], [7, 0, -1, -1], [2, 4, 0, 1]],
                                       [[0.25, 0.9, 0.5, 0.25], [0.5, 0.5, 0.3, 0.3], [0.1, 0.2, 0.3, 0.4]], 5)
    assert np.array_equal(q[0], np.float32([0, 0.25, 0, 0.75, 0]))   # padding ignored, repeats add up
    assert np.array_equal(q[1], np.float32([0.5, 0, 0, 0, 0]))       # id 7 >= V is dropped ...
    assert bad.tolist() == [False, True, False]                      # ... and marks its row
    assert np.array_equal(q[2], np.float32([0.3, 0.4, 0.1, 0, 0.2]))


def test_every_id_as_candidate_equals_the_dense_oracle():
    w = wl.rejection_chain(batch=6, m=5, vocab=257, dtype="bf16", boost=2.0, seed=31)
    rng = np.random.default_rng(1)
    perm = np.stack([rng.permutation(w.vocab) for _ in range(w.rows)]).astype(np.int32)
    probs = np.take_along_axis(w.q, perm, axis=1)
    ws = dataclasses.replace(w, kind="rejection_chain_sparse", q=None, cand_ids=perm, cand_probs=probs)
    a, b = oracle.verify_chain(w), oracle.verify_chain_sparse(ws)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_residual_reaches_outside_the_candidates():
    """P(emit v) = min(p, q)_v + (1 - sum min(p, q)) * [p - q]+_v / sum [p - q]+ = p_v, with a 2-candidate q."""
    p = np.array([0.30, 0.25, 0.20, 0.15, 0.10], dtype=np.float64)
    q, _ = oracle.scatter_candidates([[1, 3]], [[0.7, 0.3]], 5)
    q = q[0].astype(np.float64)
    acc = np.minimum(p, q)
    res = oracle.residual(p, q)
    emit = acc + (1.0 - acc.sum()) * res / res.sum()
    assert np.allclose(emit, p, atol=1e-12)
    assert res[0] > 0 and res[2] > 0 and res[4] > 0   # non-candidates keep their whole p


def test_out_of_range_candidate_flags_the_request():
    w = wl.rejection_chain_sparse(batch=3, m=3, vocab=500, K=6, pad=1, seed=9)
    ids = w.cand_ids.copy()
    ids[5, 2] = 500          # request 1, row 1 (tested)
    ids[11, 0] = 9999        # request 2's last row: never tested, not flagged
    o = oracle.verify_chain_sparse(dataclasses.replace(w, cand_ids=ids))
    assert [int(s) & 1 for s in o["status"]] == [0, 1, 0]


def test_generator_draws_drafts_from_the_candidates():
    w = wl.rejection_chain_sparse(batch=4, m=4, vocab=3000, K=16, pad=3, seed=2)
    L = w.max_len
    for b in range(w.batch):
        for j in range(L - 1):
            r = b * L + j
            assert w.verify_ids[r + 1] in w.cand_ids[r, :16]
    assert np.allclose(w.cand_probs[:, :16].astype(np.float64).sum(axis=1), 1.0, atol=1e-6)
    assert (w.cand_ids[:, 16:] == -1).all()
