"""Comparison of an implementation's verification outputs with the oracle's.

Test infrastructure only: imported by tests/, by the package smoke check and
by the benchmark's CPU-baseline leg.  The product path never imports it.

The rule (speculative decoding, [E2D] "从 EAGLE 到 DFlash 2" §1.2: accept with
probability alpha = min(1, p/q), resample the first rejection from
[p - q]_+): token decisions — accepted lengths, token ids, committed rows and
KV-commit indices, status bits — must be bit-exact.  The one exception is a
decision whose uniform lies within `tol` of its threshold (the oracle's
test_gap for an acceptance test, draw_gap for the final inverse-CDF draw):
finite precision may take it either way.  Such a request is compared exactly up
to that decision:

* final draw close, every test far: everything but the drawn token (bonus and
  its slot in out_tokens) is exact; the drawn token must be a valid id;
* first close test at step k: the first k accepted tokens and the k + 1
  committed rows are exact; what follows must be a valid verification result
  (the path continues through the given drafts / tree children, num_out =
  accept_len + 1, the last output is the bonus).

Commit lists are always checked against the implementation's own committed
rows (commit_cu is the exclusive scan of num_out; slot = row_slots[row],
position = seq_len + k), and against the oracle's for exactly compared requests.
"""
from __future__ import annotations

import numpy as np

GAP_TOL = 1e-6
KEYS = ("accept_len", "num_out", "bonus", "out_tokens", "accept_rows", "status")


def _path_valid(w, b: int, g: dict) -> list:
    """Problems with request b's result as a verification outcome of its own inputs (empty when valid)."""
    bad = []
    r = int(g["accept_len"][b])
    n = int(g["num_out"][b])
    rows = np.asarray(g["accept_rows"][b])
    toks = np.asarray(g["out_tokens"][b])
    ML = rows.shape[0]
    if not (0 <= r < ML) or n != r + 1:
        return ["accept_len %d / num_out %d out of range" % (r, n)]
    bonus = int(g["bonus"][b])
    if not (0 <= bonus < w.vocab) or int(toks[r]) != bonus:
        bad.append("bonus %d (out_tokens[r] %d)" % (bonus, int(toks[r])))
    if np.any(toks[r + 1:] != -1) or np.any(rows[r + 1:] != -1):
        bad.append("entries past num_out are not -1")
    if w.nodes:  # tree: node k+1 is a child of node k, its token is the output
        N = w.nodes
        nodes = rows[: r + 1] - b * N
        if nodes[0] != 0 or np.any((nodes < 0) | (nodes >= N)):
            return bad + ["path rows %s leave the request" % rows[: r + 1].tolist()]
        for k in range(r):
            c = int(nodes[k + 1])
            if int(w.parents[b, c]) != int(nodes[k]) or int(toks[k]) != int(w.tokens[b, c]):
                bad.append("step %d: node %d is not a child of %d carrying token %d" % (k, c, nodes[k], toks[k]))
    else:  # chain / ragged: rows start.., tokens are the drafts
        start = int(w.cu_seqlens[b])
        if r + 1 > int(w.cu_seqlens[b + 1]) - start:
            return bad + ["accept_len %d exceeds the request's drafts" % r]
        if not np.array_equal(rows[: r + 1], np.arange(start, start + r + 1)):
            bad.append("committed rows %s" % rows[: r + 1].tolist())
        if not np.array_equal(toks[:r], np.asarray(w.verify_ids[start + 1:start + 1 + r])):
            bad.append("accepted tokens are not the drafts")
    return bad


def _commit_lists_ok(w, g: dict) -> list:
    """The implementation's commit lists follow from its own num_out and committed rows."""
    bad = []
    cu = np.concatenate([[0], np.cumsum(np.asarray(g["num_out"], np.int64))])
    if not np.array_equal(np.asarray(g["commit_cu"], np.int64), cu):
        return ["commit_cu is not the exclusive scan of num_out"]
    for b in range(w.batch):
        n = int(g["num_out"][b])
        rows = np.asarray(g["accept_rows"][b][:n], np.int64)
        s = int(cu[b])
        if g.get("commit_src_slot") is not None and w.row_slots is not None and n:
            if not np.array_equal(np.asarray(g["commit_src_slot"][s:s + n]), np.asarray(w.row_slots)[rows]):
                bad.append((b, "commit_src_slot"))
        if g.get("commit_dst_pos") is not None and w.seq_lens is not None and n:
            if not np.array_equal(np.asarray(g["commit_dst_pos"][s:s + n]), int(w.seq_lens[b]) + np.arange(n)):
                bad.append((b, "commit_dst_pos"))
    return bad


def compare(w, g: dict, o: dict, tol: float = GAP_TOL, check: bool = True) -> dict:
    """Compare implementation outputs g with oracle outputs o on workload w.

    Returns counts: requests; exact (compared in full); draw_flagged (only the
    final draw within tol of a CDF edge); test_flagged (an acceptance test
    within tol: compared up to it); differ (flagged requests whose result is not
    the oracle's); mismatch (violations of the rule).  With check=True a
    mismatch raises AssertionError listing the first few.
    """
    B = w.batch
    test_gap = np.asarray(o["test_gap"], np.float64).reshape(B, -1)
    draw_gap = np.asarray(o["draw_gap"], np.float64)
    bad = []
    exact = draw_fl = test_fl = differ = 0
    for b in range(B):
        close = np.nonzero(test_gap[b] < tol)[0]
        same = all(np.array_equal(np.asarray(g[k][b]), np.asarray(o[k][b])) for k in KEYS)
        if close.size == 0 and not draw_gap[b] < tol:
            exact += 1
            for k in KEYS:
                if not np.array_equal(np.asarray(g[k][b]), np.asarray(o[k][b])):
                    bad.append((b, k, g[k][b], o[k][b]))
            continue
        differ += 0 if same else 1
        if close.size == 0:  # only the final draw is close: all but the drawn token is exact
            draw_fl += 1
            r = int(o["accept_len"][b])
            for k in ("accept_len", "num_out", "accept_rows", "status"):
                if not np.array_equal(np.asarray(g[k][b]), np.asarray(o[k][b])):
                    bad.append((b, k, g[k][b], o[k][b]))
            gt, ot = np.asarray(g["out_tokens"][b]).copy(), np.asarray(o["out_tokens"][b]).copy()
            gt[r] = ot[r] = 0
            if not np.array_equal(gt, ot):
                bad.append((b, "out_tokens before the draw", g["out_tokens"][b], o["out_tokens"][b]))
        else:  # first close test at step k0: exact up to it, valid after it
            test_fl += 1
            k0 = int(close[0])
            if int(g["accept_len"][b]) < k0:
                bad.append((b, "accept_len below the first close test", int(g["accept_len"][b]), k0))
            elif not (np.array_equal(np.asarray(g["out_tokens"][b][:k0]), np.asarray(o["out_tokens"][b][:k0])) and
                      np.array_equal(np.asarray(g["accept_rows"][b][:k0 + 1]),
                                     np.asarray(o["accept_rows"][b][:k0 + 1]))):
                bad.append((b, "prefix before the first close test", g["accept_rows"][b], o["accept_rows"][b]))
        for msg in _path_valid(w, b, g):
            bad.append((b, "invalid result: " + msg))
    if exact == B:  # nothing flagged: whole-batch equality of the commit lists
        if not np.array_equal(np.asarray(g["commit_cu"]), np.asarray(o["commit_cu"])):
            bad.append(("commit_cu",))
        n = int(o["commit_cu"][-1])
        for k in ("commit_src_slot", "commit_dst_pos"):
            if g.get(k) is not None and not np.array_equal(np.asarray(g[k][:n]), np.asarray(o[k][:n])):
                bad.append((k,))
    else:
        bad.extend(_commit_lists_ok(w, g))
    if check:
        assert not bad, "mismatches (first 5 of %d): %s" % (len(bad), bad[:5])
    return {"requests": B, "exact": exact, "draw_flagged": draw_fl, "test_flagged": test_fl,
            "flagged": draw_fl + test_fl, "differ": differ, "mismatch": len(bad)}
