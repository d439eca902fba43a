"""DSpark verify-length scheduling, restated in plain Python (fp64).

Test infrastructure only: imported by tests/, by the package smoke check and
by the benchmark's CPU-baseline leg.  The product path never imports it.

Source: "从 EAGLE 到 DFlash 2：SGLang 与 SpecForge 的投机解码训练和推理",
section 5.6.3 (the host chooses the extra draft budget K from historical
survival scores and a speed table) and section 5.6.4 (the device gives the
budget to the current best positions: global top-K by survival, ties by
position, then by request; verify length = 1 anchor + the selected drafts).
"""
from __future__ import annotations

import math
from typing import Sequence


def budget(hist_survival: Sequence[float], num_requests: int, sps: Sequence[float], eps: float = 0.0) -> int:
    """K* = argmax over K of N(K) * SPS(R + K), section 5.6.3.

    Scores below eps (and NaN) are dropped; the rest are sorted in
    descending order a_1 >= a_2 >= ...; N(K) = R + a_1 + ... + a_K predicts
    the committed tokens of a round with R + K target rows, and sps[M] is
    the speed (rounds per second) of a round with M target rows.  K stops
    where the table ends.  Equal scores keep the smaller K.
    """
    a = sorted((float(x) for x in hist_survival if not math.isnan(float(x)) and float(x) >= eps), reverse=True)
    best_k, best = 0, -math.inf
    n_hat = float(num_requests)
    for k in range(len(a) + 1):
        if k > 0:
            n_hat += a[k - 1]
        m = num_requests + k
        if m >= len(sps):
            break
        score = n_hat * float(sps[m])
        if score > best:
            best, best_k = score, k
    return best_k


def budget_table(hist_survival: Sequence[float], num_requests: int, sps: Sequence[float], eps: float = 0.0):
    """The rows of the section 5.6.3 table: (K, target rows, predicted N, SPS, predicted tokens/s)."""
    a = sorted((float(x) for x in hist_survival if not math.isnan(float(x)) and float(x) >= eps), reverse=True)
    rows, n_hat = [], float(num_requests)
    for k in range(len(a) + 1):
        if k > 0:
            n_hat += a[k - 1]
        m = num_requests + k
        if m >= len(sps):
            break
        rows.append((k, m, n_hat, float(sps[m]), n_hat * float(sps[m])))
    return rows


def selected_extra(survival: Sequence[Sequence[float]], k: int, eps: float = 0.0) -> list:
    """Drafts each request gets from the global top-k, section 5.6.4.

    Every (request r, draft position j) is one candidate with score
    survival[r][j].  Candidates are ordered by score descending, then
    position ascending, then request ascending; no token enters the order.
    The first k candidates whose score is at least eps are selected (NaN
    scores order last and are never selected).
    """
    cands = []
    for r, row in enumerate(survival):
        for j, s in enumerate(row):
            s = float(s)
            key = -math.inf if math.isnan(s) else s
            cands.append((-key, j, r, s))
    cands.sort()
    extra = [0] * len(survival)
    for rank, (_, _, r, s) in enumerate(cands):
        if rank >= k:
            break
        if not math.isnan(s) and s >= eps:
            extra[r] += 1
    return extra


def verify_lens(survival: Sequence[Sequence[float]], k: int, min_len: int = 1, max_len: int | None = None,
                eps: float = 0.0) -> list:
    """verify_len_r = clamp(1 + selected_extra_r, min_len, max_len): one anchor row plus the selected drafts."""
    extra = selected_extra(survival, k, eps)
    if max_len is None:
        max_len = 1 + max((len(row) for row in survival), default=0)
    return [min(max(1 + e, min_len), max_len) for e in extra]
