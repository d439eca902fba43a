"""Pins of the oracle's decision gaps (test_gap, draw_gap, min_gap).

The parity rule exempts a request from exact comparison from its first
decision whose uniform lies within 1e-6 of the threshold that decides it
(acceptance with probability min(1, p/q) and the residual / bonus draw by
inverse CDF, [E2D] "从 EAGLE 到 DFlash 2" §1.2 and §6.2).  So the reported
gaps decide what the GPU tests compare; a gap that came out too large would
exempt too little, one too small would exempt too much.

The pin does not recompute the gap from its formula.  It moves the decision's
own uniform and runs the oracle again: a move of (1 - eps) * gap in either
direction must leave the request's outcome unchanged, and a move just past the
gap (by min(eps * gap, 1e-5)) toward the threshold must change it.  Only uniforms in [0, 1)
are used for the first check (the domain of the caller's uniforms).
"""
import dataclasses

import numpy as np
import pytest

import oracle
from oracle import match
from reject_row_vocab_gb300 import workload as wl

EPS = 0.02
MIN_GAP = 2e-3  # perturbations of EPS * gap must stay far above fp32 spacing of the uniforms
OVERSHOOT = 1e-5  # largest step past a threshold


def _outcome(o, b):
    return (int(o["accept_len"][b]), int(o["bonus"][b]), tuple(np.asarray(o["out_tokens"][b]).tolist()))


def _check_slot(run, w, field, index_of, gaps, base):
    """Perturb uniform `field`[index_of[b]] of every request b by +-(1 -+ EPS) * gaps[b]."""
    B = w.batch
    live = np.isfinite(gaps) & (gaps > MIN_GAP) & (index_of >= 0)
    if not live.any():
        return 0
    u0 = getattr(w, field).astype(np.float64)
    flipped = np.zeros(B, bool)
    for sign in (+1.0, -1.0):
        for want_same in (True, False):
            u = u0.copy()
            moved = np.zeros(B, bool)
            for b in np.nonzero(live)[0]:
                i = index_of[b]
                # just short of the gap, or just past it (by at most 1e-5: thresholds may sit near 0 or 1)
                step = (1.0 - EPS) * gaps[b] if want_same else gaps[b] + min(EPS * gaps[b], OVERSHOOT)
                v = u0[i] + sign * step
                if want_same and not (0.0 <= v < 1.0):
                    continue
                if not want_same and v < 0.0:
                    continue
                u[i] = v
                moved[b] = True
            o = run(dataclasses.replace(w, **{field: u.astype(np.float32)}))
            for b in np.nonzero(moved)[0]:
                same = _outcome(o, b) == _outcome(base, b)
                if want_same:
                    assert same, "request %d changed under a move of %.6g < its gap %.6g" % (
                        b, (1.0 - EPS) * gaps[b], gaps[b])
                else:
                    flipped[b] |= not same
    assert np.all(flipped[live]), "requests %s did not change under a move just past their gap" % (
        np.nonzero(live & ~flipped)[0].tolist())
    return int(live.sum())


def _pin_chain(run, w, draw_field="u_final"):
    """draw_field: the uniform of the final draw (u_final[b], or u_accept of the request's last row when every
    row draws with its own uniform)."""
    base = run(w)
    B, L = w.batch, w.max_len
    tg = np.asarray(base["test_gap"]).reshape(B, L)
    dg = np.asarray(base["draw_gap"])
    assert np.array_equal(np.asarray(base["min_gap"]), np.minimum(tg.min(axis=1), dg))
    n = 0
    cu = np.asarray(w.cu_seqlens)
    for k in range(L):
        idx = np.where(k < np.diff(cu), cu[:-1] + k, -1)
        n += _check_slot(run, w, "u_accept", idx, tg[:, k], base)
    if draw_field == "u_final":
        n += _check_slot(run, w, "u_final", np.arange(B), dg, base)
    else:
        n += _check_slot(run, w, "u_accept", cu[1:] - 1, dg, base)
    return n


@pytest.mark.parametrize("V,T,sigma,seed", [(6, 1.0, 1.0, 1), (16, 0.7, 2.0, 2), (11, 1.3, 0.5, 3)])
def test_rejection_chain_gaps_are_flip_distances(V, T, sigma, seed):
    w = wl.rejection_chain(batch=120, m=4, vocab=V, dtype="f32", sigma=sigma, boost=0.0, temperature=T,
                           noise_sigma=1.0, seed=seed)
    n = _pin_chain(lambda x: oracle.verify_chain(x), w)
    assert n > 100  # most decisions were exercised


def test_residual_draw_gaps_on_sparse_weights():
    # q equal to p on most ids leaves a residual with a few positive entries: the outer CDF edges
    # (no positive weight before / after the drawn id) must not count as thresholds.
    w = wl.rejection_chain(batch=150, m=2, vocab=8, dtype="f32", sigma=2.0, boost=0.0, temperature=1.0,
                           noise_sigma=0.3, seed=5)
    n = _pin_chain(lambda x: oracle.verify_chain(x), w)
    assert n > 100
    o = oracle.verify_chain(w)
    assert np.isinf(o["draw_gap"]).any() or np.all(np.isfinite(o["draw_gap"]))


def test_single_positive_weight_has_no_draw_threshold():
    w = np.zeros(9)
    w[4] = 0.3
    for u in (0.0, 0.5, 1.0 - 2.0 ** -24):
        v, g = oracle.sample_index(w, u)
        assert v == 4 and np.isinf(g)
    w[7] = 0.1  # an upper edge appears at 0.75; nothing lies below id 4
    v, g = oracle.sample_index(w, 0.7)
    assert v == 4 and abs(g - 0.05) < 1e-12
    v, g = oracle.sample_index(w, 0.1)
    assert v == 4 and abs(g - 0.65) < 1e-12
    v, g = oracle.sample_index(w, 0.8)  # id 7: its lower edge only
    assert v == 7 and abs(g - 0.05) < 1e-12


def test_match_chain_gaps_are_flip_distances():
    w = wl.rejection_chain(batch=100, m=3, vocab=7, dtype="f32", sigma=1.0, boost=0.0, temperature=1.0,
                           noise_sigma=0.2, seed=9)
    w = dataclasses.replace(w, kind="sample_match_chain", q=None)
    n = _pin_chain(match.verify_chain_match, w, draw_field="u_accept")
    assert n > 100


def test_target_only_tree_gaps_are_flip_distances():
    # theta_single = 2 keeps the threshold on p out of reach, so every gap is a uniform's distance
    w = wl.eagle2_tree(batch=80, topk=3, depth=3, keep=8, vocab=12, mode="target_only_tree", noise_sigma=0.5,
                       temperature=1.0, seed=4)
    w = dataclasses.replace(w, threshold_single=2.0)
    run = lambda x: oracle.verify_tree(x, "target_only")  # noqa: E731
    base = run(w)
    B, N = w.batch, w.nodes
    tg = np.asarray(base["test_gap"]).reshape(B, N)
    dg = np.asarray(base["draw_gap"])
    assert np.array_equal(np.asarray(base["min_gap"]), np.minimum(tg.min(axis=1), dg))
    n = 0
    rows = np.asarray(base["accept_rows"])
    for k in range(N):  # the node at depth k of the oracle's path owns u_accept[its row]
        idx = np.where(rows[:, k] >= 0, rows[:, k], -1)
        n += _check_slot(run, w, "u_accept", idx, tg[:, k], base)
    n += _check_slot(run, w, "u_final", np.arange(B), dg, base)
    assert n > 80
