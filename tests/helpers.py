"""Small builders shared by the tests (input construction only)."""
from __future__ import annotations

import numpy as np

from reject_row_vocab_gb300.workload import Workload


def chain_workload(logits, dtype, cu, ids, q=None, T=None, ua=None, uf=None, max_len=None, kind=None,
                   row_slots=None, seq_lens=None, name="custom"):
    logits = np.ascontiguousarray(logits)
    cu = np.asarray(cu, np.int32)
    B = len(cu) - 1
    R, V = logits.shape
    lens = np.diff(cu)
    if max_len is None:
        max_len = int(max(1, lens.max())) if B else 1
    if row_slots is None:
        row_slots = np.arange(R, dtype=np.int64) + 1000
    if seq_lens is None:
        seq_lens = np.full(B, 100, np.int64)
    return Workload(kind=kind or ("rejection_ragged" if q is not None else "greedy_chain"), name=name,
                    dtype=dtype, logits=logits, batch=B, vocab=V, rows=R, max_len=int(max_len),
                    m=None, cu_seqlens=cu, verify_ids=np.asarray(ids, np.int32),
                    q=None if q is None else np.ascontiguousarray(q, np.float32),
                    temperature=None if T is None else np.asarray(T, np.float32),
                    u_accept=None if ua is None else np.asarray(ua, np.float32),
                    u_final=None if uf is None else np.asarray(uf, np.float32),
                    row_slots=np.asarray(row_slots, np.int64), seq_lens=np.asarray(seq_lens, np.int64))


def tree_workload(logits, dtype, tokens, parents, T=None, ua=None, uf=None, kind="greedy_tree",
                  th_single=1.0, th_acc=1.0, first_child=None, next_sibling=None, name="custom_tree"):
    tokens = np.asarray(tokens, np.int32)
    parents = np.asarray(parents, np.int32)
    B, N = tokens.shape
    logits = np.ascontiguousarray(logits)
    R, V = logits.shape
    assert R == B * N
    return Workload(kind=kind, name=name, dtype=dtype, logits=logits, batch=B, vocab=V, rows=R, max_len=N,
                    nodes=N, tokens=tokens, parents=parents,
                    first_child=None if first_child is None else np.asarray(first_child, np.int32),
                    next_sibling=None if next_sibling is None else np.asarray(next_sibling, np.int32),
                    temperature=None if T is None else np.asarray(T, np.float32),
                    u_accept=None if ua is None else np.asarray(ua, np.float32),
                    u_final=None if uf is None else np.asarray(uf, np.float32),
                    threshold_single=th_single, threshold_acc=th_acc,
                    row_slots=np.arange(R, dtype=np.int64) + 5000, seq_lens=np.full(B, 40, np.int64))


def chi_square_pvalue(counts, probs):
    """Pearson chi-square goodness of fit p-value (bins with tiny expectation merged)."""
    from scipy import stats
    counts = np.asarray(counts, np.float64)
    n = counts.sum()
    exp = np.asarray(probs, np.float64) * n
    keep = exp >= 5
    c = list(counts[keep])
    e = list(exp[keep])
    if (~keep).any():
        c.append(counts[~keep].sum())
        e.append(exp[~keep].sum())
    c, e = np.array(c), np.array(e)
    if len(c) < 2:
        return 1.0
    chi2 = ((c - e) ** 2 / np.maximum(e, 1e-300)).sum()
    return float(stats.chi2.sf(chi2, len(c) - 1))
