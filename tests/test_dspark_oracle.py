"""Pins of the DSpark scheduling oracle (no GPU).

The worked example of the page (budget table and device allocation) is the
golden fixture; the properties below hold for any input.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import dspark

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "dspark_scheduler_example.json")))


def _sps_list(d):
    m = max(int(k) for k in d)
    return [float(d[str(i)]) if str(i) in d else 0.0 for i in range(m + 1)]


def test_budget_table_and_k_star_match_the_page():
    g = GOLD["budget"]
    hist = [x for row in g["hist_survival"] for x in row]
    sps = _sps_list(g["sps_by_target_rows"])
    rows = dspark.budget_table(hist, g["num_requests"], sps)
    assert len(rows) == len(g["table"])
    for (k, m, n, s, tps), want in zip(rows, g["table"]):
        assert (k, m) == (want["K"], want["rows"])
        assert n == pytest.approx(want["N"], abs=1e-12)
        assert s == want["sps"]
        assert tps == pytest.approx(want["tokens_per_s"], abs=1e-9)
    assert dspark.budget(hist, g["num_requests"], sps) == g["k_star"]


def test_allocation_matches_the_page():
    g = GOLD["allocation"]
    assert dspark.selected_extra(g["survival"], g["budget"]) == g["selected_extra"]
    lens = dspark.verify_lens(g["survival"], g["budget"])
    assert lens == g["verify_lens"]
    assert sum(lens) == g["target_rows"]


def test_budget_edge_cases():
    sps = [0.0, 10.0, 9.0, 8.0]
    assert dspark.budget([], 1, sps) == 0                      # nothing to add
    assert dspark.budget([0.5, 0.5, 0.5, 0.5], 1, sps) == 2    # table ends at 3 rows
    assert dspark.budget([0.9, float("nan"), 0.01], 1, sps, eps=0.05) == 1  # NaN and sub-eps scores dropped
    # a flat speed table takes every positive score
    assert dspark.budget([0.3, 0.2, 0.1], 2, [1.0] * 10) == 3
    # equal predicted throughput keeps the smaller K: N(K) * SPS(1 + K) = 1*6 = 2*3 = 3*2 exactly
    assert dspark.budget([1.0, 1.0], 1, [0.0, 6.0, 3.0, 2.0]) == 0
    assert dspark.budget([1.0, 1.0], 1, [0.0, 5.0, 3.0, 2.0]) == 1  # K = 1 and K = 2 tie above K = 0


def test_monotone_rows_get_prefixes_and_the_budget_is_spent():
    rng = np.random.default_rng(5)
    for _ in range(200):
        R, D = int(rng.integers(1, 7)), int(rng.integers(1, 9))
        conf = rng.choice([0.5, 0.8, 0.9, 1.0], size=(R, D))    # repeated values force ties
        surv = np.cumprod(conf, axis=1)
        k = int(rng.integers(0, R * D + 2))
        extra = dspark.selected_extra(surv.tolist(), k)
        assert sum(extra) == min(k, R * D)
        # a pairwise rank count (score, then position, then request) selects
        # exactly the first extra[r] positions of every row: prefixes only
        for r in range(R):
            for j in range(D):
                s = surv[r, j]
                better = sum(1 for rr in range(R) for jj in range(D)
                             if surv[rr, jj] > s or (surv[rr, jj] == s and (jj < j or (jj == j and rr < r))))
                assert (better < k) == (j < extra[r])


def test_ties_break_by_position_then_request():
    s = [[0.5, 0.5], [0.5, 0.5]]
    assert dspark.selected_extra(s, 1) == [1, 0]   # (pos 0, req 0) first
    assert dspark.selected_extra(s, 2) == [1, 1]   # then (pos 0, req 1)
    assert dspark.selected_extra(s, 3) == [2, 1]   # then (pos 1, req 0)
    assert dspark.verify_lens(s, 4, max_len=2) == [2, 2]
    assert dspark.verify_lens([[float("nan"), 0.2]], 2, eps=0.1) == [2]


# ---------------------------------------------------------------------------
# The library's host budget (no GPU) against the oracle and the page
# ---------------------------------------------------------------------------

def _lib():
    from reject_row_vocab_gb300 import _build, specverify
    _build.build()
    return specverify


def test_library_budget_matches_the_page_and_the_oracle():
    sv = _lib()
    g = GOLD["budget"]
    hist = [x for row in g["hist_survival"] for x in row]
    sps = _sps_list(g["sps_by_target_rows"])
    assert sv.dspark_budget(hist, g["num_requests"], sps) == g["k_star"]
    rng = np.random.default_rng(11)
    for _ in range(300):
        n = int(rng.integers(0, 40))
        hist = rng.choice([0.0, 0.1, 0.25, 0.5, 0.75, 1.0, float("nan")], size=n).astype(np.float32)
        R = int(rng.integers(0, 8))
        sps = np.sort(rng.uniform(1, 100, size=int(rng.integers(1, 30))).astype(np.float32))[::-1].copy()
        eps = float(rng.choice([0.0, 0.2]))
        # the oracle in fp64 over the same fp32 inputs
        want = dspark.budget(hist.astype(np.float64).tolist(), R, sps.astype(np.float64).tolist(), eps)
        assert sv.dspark_budget(hist, R, sps, eps) == want
    # exact ties keep the smaller K in the library too
    assert sv.dspark_budget(np.array([1.0, 1.0], np.float32), 1, np.array([0.0, 6.0, 3.0, 2.0], np.float32)) == 0
    assert sv.dspark_budget(np.array([1.0, 1.0], np.float32), 1, np.array([0.0, 5.0, 3.0, 2.0], np.float32)) == 1


def test_library_scheduler_host_validation():
    import ctypes
    sv = _lib()
    lib = sv.load_library()
    k = ctypes.c_int32()
    assert lib.spec_verify_dspark_budget(None, 0, 1, None, 0, 0.0, None) == 1        # SV_ERR_NULL_ARG
    assert lib.spec_verify_dspark_budget(None, -1, 1, None, 0, 0.0, ctypes.byref(k)) == 2
    assert lib.spec_verify_dspark_budget(None, 0, 3, None, 0, 0.0, ctypes.byref(k)) == 0 and k.value == 0
    fake = ctypes.c_void_p(0x100000)
    ws = ctypes.c_void_p(0x100000)
    f = lib.spec_verify_dspark_verify_lens
    assert f(fake, 2, 3, 2, 1, 1, 4, 0.0, fake, ws, 256, None) == 2          # ld < D
    assert f(fake, 2, 3, 3, -1, 1, 4, 0.0, fake, ws, 256, None) == 2         # negative budget
    assert f(fake, 2, 3, 3, 1, 0, 4, 0.0, fake, ws, 256, None) == 2          # min_len < 1
    assert f(fake, 2, 3, 3, 1, 3, 2, 0.0, fake, ws, 256, None) == 2          # max_len < min_len
    assert f(None, 2, 3, 3, 1, 1, 4, 0.0, fake, ws, 256, None) == 1          # survival NULL
    assert f(fake, 2, 3, 3, 1, 1, 4, 0.0, fake, None, 256, None) == 6        # no workspace
    assert f(fake, 2, 3, 3, 1, 1, 4, 0.0, fake, ctypes.c_void_p(0x100010), 256, None) == 6  # misaligned
    assert f(None, 0, 3, 3, 1, 1, 4, 0.0, None, None, 0, None) == 0          # no requests: nothing to do
