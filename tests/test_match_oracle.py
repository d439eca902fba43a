"""Pins of the sample-then-match oracle (no GPU)."""
import dataclasses

import numpy as np

import oracle
from oracle import match
from reject_row_vocab_gb300 import workload as wl


def _small(T=0.9, seed=3, batch=1, m=3, vocab=12):
    return wl.rejection_chain(batch=batch, m=m, vocab=vocab, dtype="f32", boost=2.0, temperature=T, seed=seed,
                              noise_sigma=0.3)


def test_greedy_requests_equal_the_greedy_chain_oracle():
    w = wl.rejection_chain(batch=7, m=5, vocab=300, dtype="bf16", boost=3.0, seed=8)
    wg = dataclasses.replace(w, temperature=np.zeros(w.batch, np.float32))
    a = match.verify_chain_match(wg)
    b = oracle.verify_chain(wg, greedy_all=True)
    for k in ("accept_len", "num_out", "out_tokens", "bonus", "accept_rows", "commit_cu", "status"):
        assert np.array_equal(a[k], b[k]), k


def test_accept_length_is_the_cumulative_product_of_match_probabilities():
    """P(accept_len >= k) = prod_{j<k} p_j(d_{j+1}) over independent uniforms (the 'cumprod' loop)."""
    w = _small()
    L = w.max_len
    p = [oracle.row_probs(w.logits, w.dtype, j, float(w.temperature[0])) for j in range(L)]
    match_p = [p[j][int(w.verify_ids[j + 1])] for j in range(L - 1)]
    want = np.cumprod([1.0] + match_p)          # P(s >= k), k = 0 .. L-1
    rng = np.random.default_rng(0)
    n = 20000
    counts = np.zeros(L)
    for _ in range(n):
        wu = dataclasses.replace(w, u_accept=rng.random(L).astype(np.float32))
        s = int(match.verify_chain_match(wu)["accept_len"][0])
        counts[:s + 1] += 1
    got = counts / n
    sd = np.sqrt(want * (1 - want) / n) + 1e-12
    assert np.all(np.abs(got - want) < 5 * sd + 1e-3), (got, want)


def test_first_emitted_token_follows_the_target():
    """Lossless: the first emitted token (the draft if it matched, else the sample) is distributed as p_0."""
    w = _small(seed=5, vocab=8)
    p0 = oracle.row_probs(w.logits, w.dtype, 0, float(w.temperature[0]))
    rng = np.random.default_rng(1)
    n = 20000
    hist = np.zeros(w.vocab)
    for _ in range(n):
        wu = dataclasses.replace(w, u_accept=rng.random(w.max_len).astype(np.float32))
        hist[int(match.verify_chain_match(wu)["out_tokens"][0, 0])] += 1
    exp = p0 * n
    keep = exp > 5
    chi2 = float((((hist - exp) ** 2) / np.maximum(exp, 1e-12))[keep].sum())
    assert chi2 < 40.0, (chi2, hist, exp)   # ~ chi-square with <= 7 degrees of freedom


def test_bad_draft_id_and_unusable_rows():
    w = _small(batch=3, m=3, vocab=20, seed=9)
    ids = w.verify_ids.copy()
    ids[1] = 999                     # request 0, row 0 tests an out-of-range id
    x = w.logits.copy()
    x[4 + 0, :] = -np.inf            # request 1, row 0 has no usable logit
    o = match.verify_chain_match(dataclasses.replace(w, verify_ids=ids, logits=x))
    assert o["accept_len"][0] == 0 and int(o["status"][0]) & 1
    assert int(o["status"][1]) & 2 and o["accept_len"][1] == 0 and o["bonus"][1] == -1
