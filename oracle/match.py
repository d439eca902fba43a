"""Verification by independent target sampling and prefix match, restated in
plain Python over the fp64 oracle's row probabilities and inverse-CDF sampler.

Test infrastructure only: imported by tests/, by the package smoke check and
by the benchmark's CPU-baseline leg.  The product path never imports it.

Source: "从 EAGLE 到 DFlash 2：SGLang 与 SpecForge 的投机解码训练和推理",
sections 1.2 (independent target sampling followed by prefix matching is a
verification of its own, distinct from p/q rejection) and 8.1 / the DFlash
inference loop (sample the target's posterior at every block position, the
accept length is the longest prefix where draft and sample agree — the
cumulative product of matches — and the first mismatching position takes the
posterior sample).  Row j of a request is sampled by inverse CDF with the
caller's uniform u[row]; greedy requests take the argmax instead.
"""
from __future__ import annotations

import numpy as np

import oracle

NONFINITE = 2
TOKEN_RANGE = 1


def _sampling(T: float) -> bool:
    return 1e-30 <= T < float("inf")


def verify_chain_match(w) -> dict:
    """Outputs with the chain oracle's keys for a fixed-length or ragged chain workload."""
    B, V, ML = w.batch, w.vocab, w.max_len
    cu = np.asarray(w.cu_seqlens, dtype=np.int64)
    ids = np.asarray(w.verify_ids)
    st_all = oracle.row_stats(w.logits, w.dtype)
    o = {"accept_len": np.zeros(B, np.int32), "num_out": np.zeros(B, np.int32),
         "out_tokens": np.full((B, ML), -1, np.int32), "bonus": np.full(B, -1, np.int32),
         "accept_rows": np.full((B, ML), -1, np.int32), "commit_cu": np.zeros(B + 1, np.int32),
         "commit_src_slot": np.full(max(w.rows, 1), -1, np.int64),
         "commit_dst_pos": np.full(max(w.rows, 1), -1, np.int64),
         "status": np.zeros(B, np.uint32), "min_gap": np.full(B, np.inf),
         "test_gap": np.full((B, ML), np.inf), "draw_gap": np.full(B, np.inf)}
    for b in range(B):
        start, L = int(cu[b]), int(cu[b + 1] - cu[b])
        T = float(w.temperature[b]) if w.temperature is not None else 0.0
        status, gap, s, tok = 0, np.inf, L - 1, -1
        for j in range(L):
            row = start + j
            if int(st_all["flags"][row]) & NONFINITE:
                status |= NONFINITE
            if int(st_all["argmax"][row]) < 0:  # no usable logit: stop here, no token
                status |= NONFINITE
                s, tok = j, -1
                break
            g = np.inf
            if _sampling(T):
                p = oracle.row_probs(w.logits, w.dtype, row, T)
                t, g = oracle.sample_index(p, float(w.u_accept[row]))
                gap = min(gap, g)
            else:
                t = int(st_all["argmax"][row])
            if j == L - 1:  # the last row's draw only emits a token
                o["draw_gap"][b] = g
                s, tok = j, int(t)
                break
            # a tested row's draw decides the match and, at a mismatch, the emitted token
            o["test_gap"][b, j] = g
            d = int(ids[row + 1])
            if d < 0 or d >= V:
                status |= TOKEN_RANGE
                s, tok = j, int(t)
                break
            if d != t:
                s, tok = j, int(t)
                break
        o["accept_len"][b] = s
        o["num_out"][b] = s + 1
        o["out_tokens"][b, :s] = ids[start + 1:start + 1 + s]
        o["out_tokens"][b, s] = tok
        o["accept_rows"][b, :s + 1] = np.arange(start, start + s + 1)
        o["bonus"][b] = tok
        o["status"][b] = status
        o["min_gap"][b] = gap
    o["commit_cu"][1:] = np.cumsum(o["num_out"])
    for b in range(B):
        for k in range(int(o["num_out"][b])):
            dst = int(o["commit_cu"][b]) + k
            row = int(o["accept_rows"][b, k])
            if w.row_slots is not None:
                o["commit_src_slot"][dst] = w.row_slots[row]
            if w.seq_lens is not None:
                o["commit_dst_pos"][dst] = w.seq_lens[b] + k
    return o
