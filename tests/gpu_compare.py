"""Comparison of the CUDA path with the oracle on the same seeded inputs.

The rule itself (what is exact, what a near-threshold decision exempts) lives
in oracle/parity.py; this module runs the matching oracle and keeps a record of
every comparison, which tests/conftest.py prints at the end of the run.
"""
from __future__ import annotations

import os

import oracle
from oracle.parity import GAP_TOL, compare as _compare

# (workload name, counts) of every comparison made in this process
REPORT: list = []


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


def compare(w, g: dict, o: dict, tol: float = GAP_TOL) -> dict:
    """Compare and record; raises on any violation of the parity rule."""
    res = _compare(w, g, o, tol=tol, check=True)
    REPORT.append((w.name, res))
    return res


def flag_bound(batch: int, frac: float) -> int:
    """Most flagged requests a batch may have before the count itself is a failure."""
    return max(2, int(frac * batch + 0.999))
