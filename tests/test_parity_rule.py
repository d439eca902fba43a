"""The parity rule (oracle/parity.py) on outputs doctored on the CPU.

A copy of the oracle's own outputs stands in for an implementation's: the rule
must accept it unchanged, refuse any change to a decision that is far from its
threshold, and allow a different outcome only from the first near-threshold
decision on — and then only a valid one.
"""
import copy
import dataclasses

import numpy as np
import pytest

import oracle
from oracle.parity import compare
from reject_row_vocab_gb300 import workload as wl


def _chain():
    return wl.rejection_chain(batch=24, m=4, vocab=40, dtype="f32", sigma=2.0, boost=0.0, temperature=0.9,
                              noise_sigma=1.0, seed=31)


def _edge_uniform(w, o, b):
    """A uniform 1e-8 above the upper CDF edge that request b's final draw is closest to."""
    L = w.max_len
    r = int(o["accept_len"][b])
    s = b * L + r
    p = oracle.row_probs(w.logits, w.dtype, s, float(w.temperature[b]))
    wts = np.maximum(0.0, p - w.q[s].astype(np.float64)) if r < L - 1 else p
    cdf = np.cumsum(wts) / wts.sum()
    v = int(o["bonus"][b])
    return float(cdf[v]) + 1e-8


def _recommit(w, g):
    """Commit offsets and lists made consistent with g's committed rows."""
    g["commit_cu"] = np.concatenate([[0], np.cumsum(g["num_out"])]).astype(np.int32)
    n = int(g["commit_cu"][-1])
    rows = np.concatenate([g["accept_rows"][i, :g["num_out"][i]] for i in range(w.batch)])
    g["commit_src_slot"][:n] = w.row_slots[rows]
    g["commit_dst_pos"][:n] = np.concatenate([w.seq_lens[i] + np.arange(g["num_out"][i]) for i in range(w.batch)])


def test_identical_outputs_are_exact():
    w = _chain()
    o = oracle.verify_chain(w)
    res = compare(w, copy.deepcopy(o), o)
    assert res["exact"] + res["flagged"] == w.batch and res["mismatch"] == 0 and res["differ"] == 0


@pytest.mark.parametrize("key", ["accept_len", "bonus", "status"])
def test_change_far_from_any_threshold_is_a_mismatch(key):
    w = _chain()
    o = oracle.verify_chain(w)
    b = int(np.nonzero(o["min_gap"] > 1e-3)[0][0])
    g = copy.deepcopy(o)
    g[key][b] += 1
    with pytest.raises(AssertionError):
        compare(w, g, o)
    assert compare(w, g, o, check=False)["mismatch"] >= 1


def test_close_draw_exempts_only_the_drawn_token():
    w = _chain()
    o = oracle.verify_chain(w)
    b = int(np.nonzero(np.isfinite(o["draw_gap"]) & (o["test_gap"].min(axis=1) > 1e-3))[0][0])
    uf = w.u_final.astype(np.float64).copy()
    uf[b] = _edge_uniform(w, o, b)
    w2 = dataclasses.replace(w, u_final=uf.astype(np.float32))
    o2 = oracle.verify_chain(w2)
    assert o2["draw_gap"][b] < 1e-6 <= o2["test_gap"][b].min()
    g = copy.deepcopy(o2)
    r = int(g["accept_len"][b])
    other = (int(g["bonus"][b]) + 1) % w.vocab
    g["bonus"][b] = other
    g["out_tokens"][b, r] = other
    res = compare(w2, g, o2)
    assert res["draw_flagged"] >= 1 and res["differ"] == 1 and res["mismatch"] == 0
    g["accept_len"][b] = max(0, r - 1) if r else 1  # the accepted length is still certain
    assert compare(w2, g, o2, check=False)["mismatch"] >= 1
    g = copy.deepcopy(o2)
    g["bonus"][b] = g["out_tokens"][b, r] = other
    g["status"][b] |= 16  # a valid path with a wrong status bit: the status stays exact too
    assert compare(w2, g, o2, check=False)["mismatch"] >= 1
    g = copy.deepcopy(o2)
    g["bonus"][b] = g["out_tokens"][b, r] = w.vocab  # the drawn token must be a valid id
    assert compare(w2, g, o2, check=False)["mismatch"] >= 1


def test_close_test_exempts_from_that_step_on():
    w = _chain()
    o = oracle.verify_chain(w)
    L = w.max_len
    # a request that accepted its first draft; put row 1's uniform on its threshold p/q
    cand = np.nonzero((o["accept_len"] >= 2) & (o["min_gap"] > 1e-3))[0]
    b = int(cand[0])
    row = b * L + 1
    d = int(w.verify_ids[row + 1])
    p = oracle.row_probs(w.logits, w.dtype, row, float(w.temperature[b]))[d]
    ua = w.u_accept.astype(np.float64).copy()
    ua[row] = p / float(w.q[row, d]) - 1e-8
    assert 0.0 < ua[row] < 1.0
    w2 = dataclasses.replace(w, u_accept=ua.astype(np.float32))
    o2 = oracle.verify_chain(w2)
    assert o2["test_gap"][b, 1] < 1e-6 and o2["test_gap"][b, 0] > 1e-6
    # a valid outcome that rejects at step 1 instead: prefix of one accepted draft, new correction token
    g = copy.deepcopy(o2)
    g["accept_len"][b], g["num_out"][b] = 1, 2
    g["out_tokens"][b] = -1
    g["out_tokens"][b, 0] = w.verify_ids[b * L + 1]
    g["out_tokens"][b, 1] = g["bonus"][b] = 3
    g["accept_rows"][b] = -1
    g["accept_rows"][b, :2] = [b * L, b * L + 1]
    _recommit(w, g)
    res = compare(w2, g, o2)
    assert res["test_flagged"] == 1 and res["differ"] == 1 and res["mismatch"] == 0
    # rejecting at step 0 contradicts a certain decision
    bad = copy.deepcopy(g)
    bad["accept_len"][b], bad["num_out"][b] = 0, 1
    assert compare(w2, bad, o2, check=False)["mismatch"] >= 1
    # ... even as a valid verification of its own (one correction token at row 0, consistent commit lists)
    bad = copy.deepcopy(g)
    bad["accept_len"][b], bad["num_out"][b] = 0, 1
    bad["out_tokens"][b] = -1
    bad["out_tokens"][b, 0] = bad["bonus"][b] = 3
    bad["accept_rows"][b] = -1
    bad["accept_rows"][b, 0] = b * L
    _recommit(w, bad)
    assert compare(w2, bad, o2, check=False)["mismatch"] >= 1
    # a token that is not the draft at an accepted row is invalid
    bad = copy.deepcopy(g)
    bad["out_tokens"][b, 0] += 1
    assert compare(w2, bad, o2, check=False)["mismatch"] >= 1
    # commit lists must follow the implementation's own committed rows
    bad = copy.deepcopy(g)
    bad["commit_dst_pos"][0] += 1
    assert compare(w2, bad, o2, check=False)["mismatch"] >= 1
