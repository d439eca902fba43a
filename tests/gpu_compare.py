"""Comparison of the CUDA path with the oracle on the same seeded inputs."""
from __future__ import annotations

import os

import numpy as np

import oracle

# A decision whose uniform lies within this distance of its threshold (|u - p/q|,
# |u - c/theta|, CDF edges of the sampled index) may legitimately go either way
# in finite precision; such requests are counted and reported, not compared.
GAP_TOL = 1e-6
KEYS = ("accept_len", "num_out", "bonus", "out_tokens", "accept_rows", "status")


def oracle_outputs(w, use_lists=False):
    threads = min(32, os.cpu_count() or 1)
    if w.kind == "greedy_chain":
        return oracle.verify_chain(w, greedy_all=True, threads=threads)
    if w.kind in ("rejection_chain", "rejection_ragged"):
        return oracle.verify_chain(w, threads=threads)
    if w.kind == "rejection_chain_sparse":
        return oracle.verify_chain_sparse(w, threads=threads)
    if w.kind == "sample_match_chain":
        from oracle import match
        return match.verify_chain_match(w)
    if w.kind == "greedy_tree":
        return oracle.verify_tree(w, "greedy", threads=threads, use_lists=use_lists)
    return oracle.verify_tree(w, "target_only", threads=threads, use_lists=use_lists)


def compare(w, g: dict, o: dict, gap_tol: float = GAP_TOL) -> dict:
    """Bit-exact comparison of every unflagged request; returns counts."""
    B = w.batch
    flagged = o["min_gap"] < gap_tol
    bad = []
    for b in range(B):
        if flagged[b]:
            continue
        for k in KEYS:
            if not np.array_equal(np.asarray(g[k][b]), np.asarray(o[k][b])):
                bad.append((b, k, g[k][b], o[k][b]))
    assert not bad, "mismatches on unflagged requests (first 5): %s" % bad[:5]
    # commit lists: whole-batch equality when nothing is flagged, else per request
    if not flagged.any():
        assert np.array_equal(g["commit_cu"], o["commit_cu"])
        n = int(o["commit_cu"][-1])
        for k in ("commit_src_slot", "commit_dst_pos"):
            if k in g and g[k] is not None:
                assert np.array_equal(g[k][:n], o[k][:n]), k
    else:
        for b in range(B):
            if flagged[b]:
                continue
            n = int(o["num_out"][b])
            gs, os_ = int(g["commit_cu"][b]), int(o["commit_cu"][b])
            for k in ("commit_src_slot", "commit_dst_pos"):
                if k in g and g[k] is not None:
                    assert np.array_equal(g[k][gs:gs + n], o[k][os_:os_ + n]), (b, k)
    return {"requests": B, "flagged": int(flagged.sum()),
            "differ_flagged": int(sum(not np.array_equal(g["bonus"][b], o["bonus"][b]) or
                                      g["accept_len"][b] != o["accept_len"][b] for b in range(B) if flagged[b]))}
