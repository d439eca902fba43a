"""Pins for the fp64 oracle: what the pages and the mathematics fix, independent of the oracle's code.

Each test exercises the oracle through its C entry points and checks it
against something other than itself: a worked example printed on the pages,
an identity, a library routine (scipy softmax, numpy argmax), brute force on
tiny inputs, or a chi-square test of the output law.
"""
import itertools
import json
import os

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from reject_row_vocab_gb300 import workload as wl
from tests.helpers import chain_workload, chi_square_pvalue, tree_workload

GOLD = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# Worked examples printed on the pages
# ---------------------------------------------------------------------------


def _worked():
    with open(os.path.join(GOLD, "worked_example_commit.json")) as f:
        return json.load(f)


def test_worked_example_greedy_commit():
    g = _worked()
    ids = g["token_ids"]
    V = 16
    inp = [ids[t] for t in g["verify_input"]]
    lg = np.full((len(inp), V), -1.0, np.float32)
    for j, t in enumerate(g["row_argmax"]):
        lg[j, ids[t]] = 5.0
    w = chain_workload(lg, "f32", [0, len(inp)], inp, seq_lens=[g["seq_len_before"]])
    o = oracle.verify_chain(w, greedy_all=True)
    e = g["expected"]
    assert o["accept_len"][0] == e["accept_len"]
    assert o["num_out"][0] == e["num_out"]
    assert list(o["out_tokens"][0, :3]) == [ids[t] for t in e["out_tokens"]]
    assert list(o["out_tokens"][0, 3:]) == [-1, -1]
    rows = o["accept_rows"][0, :3]
    assert [inp[r] for r in rows] == [ids[t] for t in e["committed_rows_input_tokens"]]
    assert list(o["commit_dst_pos"][:3]) == e["commit_dst_pos"]
    assert list(o["commit_src_slot"][:3]) == list(w.row_slots[rows])
    assert list(o["commit_cu"]) == [0, 3]
    assert o["bonus"][0] == ids[e["next_anchor"]]

    v4 = g["verify_len_4_variant"]
    inp4 = [ids[t] for t in v4["verify_input"]]
    w4 = chain_workload(lg[:4], "f32", [0, 4], inp4)
    o4 = oracle.verify_chain(w4, greedy_all=True)
    assert list(o4["out_tokens"][0, :3]) == [ids[t] for t in v4["expected_out_tokens"]]
    assert o4["num_out"][0] == v4["expected_num_out"]


def test_worked_example_rejection_commit():
    """Same round under p/q rejection: spiky target rows make every decision certain."""
    g = _worked()
    ids = g["token_ids"]
    V = 16
    inp = [ids[t] for t in g["verify_input"]]
    lg = np.zeros((5, V), np.float32)
    for j, t in enumerate(g["row_argmax"]):
        lg[j, ids[t]] = 40.0
    q = np.zeros((5, V), np.float32)
    for j in range(4):
        q[j, inp[j + 1]] = 1.0  # one-hot proposal at the draft actually sent
    w = chain_workload(lg, "f32", [0, 5], inp, q=q, T=[1.0], ua=[0.5] * 5, uf=[0.5],
                       seq_lens=[g["seq_len_before"]])
    o = oracle.verify_chain(w)
    assert o["accept_len"][0] == 2
    assert list(o["out_tokens"][0, :3]) == [ids["E"], ids["F"], ids["X"]]
    assert list(o["commit_dst_pos"][:3]) == [3, 4, 5]


def test_ragged_offsets_from_verify_lens():
    with open(os.path.join(GOLD, "ragged_offsets.json")) as f:
        g = json.load(f)
    lens = g["verify_lens"]
    R = sum(lens)
    V = 8
    rng = np.random.default_rng(0)
    lg = rng.standard_normal((R, V)).astype(np.float32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    ids = rng.integers(0, V, R).astype(np.int32)
    for b in range(len(lens)):  # every draft equals its row's argmax: all accepted
        for j in range(lens[b] - 1):
            ids[cu[b] + j + 1] = np.argmax(lg[cu[b] + j])
    w = chain_workload(lg, "f32", cu, ids)
    o = oracle.verify_chain(w, greedy_all=True)
    assert list(o["commit_cu"]) == g["expected_offsets"]
    assert o["commit_cu"][-1] == g["expected_rows"]
    assert int(o["accept_len"].sum()) == g["expected_draft_budget"]
    assert list(o["num_out"]) == lens  # all accepted: m+1 outputs per request


# ---------------------------------------------------------------------------
# Greedy verification reproduces token-by-token greedy decoding
# ---------------------------------------------------------------------------


def _toy_target(prefix, V):
    """A deterministic toy target: integer-valued logits keyed by the prefix (ties are common)."""
    h = np.random.default_rng(abs(hash(tuple(prefix))) % (2 ** 63))
    return h.integers(0, 6, V).astype(np.float32)


def test_greedy_chain_equals_token_by_token_decoding():
    V, m, trials = 11, 5, 400
    rng = np.random.default_rng(7)
    rows, ids, cu, truth = [], [], [0], []
    for _ in range(trials):
        prefix = list(rng.integers(0, V, rng.integers(1, 5)))
        a = int(np.argmax(_toy_target(prefix, V)))
        ctx = prefix + [a]
        cont = []
        for _ in range(m + 1):
            x = int(np.argmax(_toy_target(ctx + cont, V)))  # first occurrence = lowest index
            cont.append(x)
        drafts = [c if rng.random() < 0.75 else int(rng.integers(0, V)) for c in cont[:m]]
        seq = [a] + drafts
        for j in range(m + 1):
            rows.append(_toy_target(ctx + drafts[:j], V))
        ids.extend(seq)
        cu.append(cu[-1] + m + 1)
        r = 0
        while r < m and drafts[r] == cont[r]:
            r += 1
        truth.append((r, cont[: r + 1]))
    w = chain_workload(np.stack(rows), "f32", cu, ids)
    o = oracle.verify_chain(w, greedy_all=True)
    n_all = 0
    for b, (r, toks) in enumerate(truth):
        assert o["accept_len"][b] == r
        assert list(o["out_tokens"][b, : r + 1]) == toks
        n_all += r == m
        if r == m:
            assert o["num_out"][b] == m + 1
    assert n_all > 0


def test_row_stats_match_library_routines():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((6, 300)) * 3).astype(np.float32)
    x[2, 17] = x[2, 200] = 50.0  # a tie: lowest index wins
    bits = wl.f32_to_bf16_bits(x)
    for dtype, arr, val in (("f32", x, x), ("bf16", bits, wl.bf16_bits_to_f32(bits))):
        T = np.linspace(0.5, 1.5, 6).astype(np.float32)
        probe = rng.integers(0, 300, 6).astype(np.int32)
        s = oracle.row_stats(arr, dtype, row_temp=T, probe=probe)
        v64 = val.astype(np.float64)
        assert np.array_equal(s["argmax"], np.argmax(v64, axis=1))
        assert np.array_equal(s["max"], v64.max(axis=1))
        for r in range(6):
            p = softmax(v64[r] / float(T[r]))
            assert abs(s["p"][r] - p[probe[r]]) < 1e-13
            assert np.allclose(oracle.row_probs(arr, dtype, r, float(T[r])), p, rtol=1e-12, atol=1e-15)
            assert abs(s["z"][r] - np.exp((v64[r] - v64[r].max()) / float(T[r])).sum()) < 1e-9 * s["z"][r]
    assert s["argmax"][2] == 17


def test_row_stats_nonfinite_entries():
    """NaN and +inf are left out of the maximum, the argmax and Z and flag their row (bit 2); -inf is an ordinary
    entry of weight 0; a row of -inf only has no argmax.  Checked against numpy over the remaining entries."""
    x = np.array([[0.5, np.nan, 2.0, -1.0],
                  [np.inf, 1.0, 3.0, 3.0],
                  [-np.inf, -np.inf, -np.inf, -np.inf],
                  [0.0, -np.inf, 1.0, 0.25]], np.float32)
    T = np.full(4, 0.7, np.float32)
    s = oracle.row_stats(x, "f32", row_temp=T)
    assert list(s["flags"]) == [2, 2, 0, 0]
    assert list(s["argmax"]) == [2, 2, -1, 2]
    for r in (0, 1, 3):
        keep = np.isfinite(x[r]) | (x[r] == -np.inf)
        v = x[r][keep].astype(np.float64)
        assert s["max"][r] == v.max()
        assert abs(s["z"][r] - np.exp((v - v.max()) / float(T[r])).sum()) < 1e-12 * s["z"][r]


# ---------------------------------------------------------------------------
# Rejection test, residual, sampler
# ---------------------------------------------------------------------------


def test_accept_set_is_interval_of_length_alpha():
    grid = np.arange(4096) / 4096.0
    for p, q in ((0.3, 0.6), (0.6, 0.3), (0.25, 0.25), (1e-3, 0.5), (0.0, 0.2), (0.7, 1.0)):
        acc = np.array([oracle.accept(p, q, u) for u in grid])
        # accepted uniforms form a prefix [0, alpha) of [0,1)
        assert not np.any(np.diff(acc.astype(int)) > 0)
        alpha = min(1.0, p / q)
        assert abs(acc.mean() - alpha) <= 1.0 / 4096 + 1e-12


def test_sampler_is_inverse_cdf():
    rng = np.random.default_rng(11)
    n_grid = 1 << 14
    grid = (np.arange(n_grid) + 0.5) / n_grid
    for V in (1, 2, 3, 7, 16):
        for _ in range(5):
            w = rng.random(V) * (rng.random(V) < 0.7)
            if w.sum() == 0:
                w[rng.integers(V)] = 1.0
            picks = np.array([oracle.sample_index(w, u)[0] for u in grid])
            assert np.all(np.diff(picks) >= 0)  # monotone in u
            freq = np.bincount(picks, minlength=V) / n_grid
            assert np.allclose(freq, w / w.sum(), atol=1.0 / n_grid + 1e-12)
            assert np.all(w[np.unique(picks)] > 0)
    assert oracle.sample_index(np.zeros(4), 0.3)[0] == -1
    # u = 0 picks the first positive weight
    assert oracle.sample_index(np.array([0.0, 0.0, 2.0, 1.0]), 0.0)[0] == 2


def test_accept_plus_residual_mass_equals_target():
    """min(p,q) + (1 - sum min(p,q)) * [p-q]_+ / sum [p-q]_+ == p  (the lossless identity)."""
    rng = np.random.default_rng(5)
    for V in (2, 5, 16, 300):
        x = (rng.standard_normal((1, V)) * 2).astype(np.float32)
        T = 0.7
        p = oracle.row_probs(x, "f32", 0, T)
        q = rng.dirichlet(np.ones(V)).astype(np.float32)
        qd = q.astype(np.float64)
        w = oracle.residual(p, q)
        alpha = np.array([np.mean([oracle.accept(p[d], qd[d], u) for u in (np.arange(512) + 0.5) / 512])
                          for d in range(min(V, 16))])
        assert np.allclose(alpha, np.minimum(1.0, p[:16] / qd[:16]), atol=1.0 / 512)
        acc_mass = np.minimum(p, qd)
        law = acc_mass + (1.0 - acc_mass.sum()) * w / w.sum()
        assert np.allclose(law, p, atol=1e-12)
        # E_{d~q}[alpha(d)] = sum min(p,q) = (sum p + sum q - sum |p-q|) / 2  (= 1 - TV when normalised)
        ea = np.sum(qd * np.minimum(1.0, p / qd))
        assert abs(ea - 0.5 * (p.sum() + qd.sum() - np.abs(p - qd).sum())) < 1e-12


# ---------------------------------------------------------------------------
# Output law of the whole chain (chi-square), special proposals
# ---------------------------------------------------------------------------


def _chain_law_case(n=60000, V=8, seed=21, q_mode="random"):
    rng = np.random.default_rng(seed)
    L = 3
    base = (rng.standard_normal((L, V)) * 1.5).astype(np.float32)
    T = 0.9
    p = [softmax(base[j].astype(np.float64) / np.float64(np.float32(T))) for j in range(L)]
    if q_mode == "random":
        qs = [rng.dirichlet(np.ones(V)).astype(np.float32) for _ in range(L)]
    else:  # q equals p up to fp32 rounding
        qs = [pj.astype(np.float32) for pj in p]
    lg = np.tile(base, (n, 1))
    q = np.tile(np.stack(qs), (n, 1))
    ids = np.zeros(n * L, np.int32)
    for j in range(L - 1):
        qd = qs[j].astype(np.float64)
        ids[np.arange(n) * L + j + 1] = rng.choice(V, size=n, p=qd / qd.sum())
    ua = wl.uniforms(rng, n * L)
    if q_mode != "random":
        ua = np.minimum(ua, np.float32(0.999))
    uf = wl.uniforms(rng, n)
    cu = (np.arange(n + 1) * L).astype(np.int32)
    w = chain_workload(lg, "f32", cu, ids, q=q, T=np.full(n, T, np.float32), ua=ua, uf=uf)
    return w, p, qs


def test_rejection_chain_output_law_chi_square():
    w, p, qs = _chain_law_case()
    o = oracle.verify_chain(w, threads=4)
    V = w.vocab
    first = o["out_tokens"][:, 0]
    assert chi_square_pvalue(np.bincount(first, minlength=V), p[0]) > 1e-4
    m1 = o["accept_len"] >= 1
    assert chi_square_pvalue(np.bincount(o["out_tokens"][m1, 1], minlength=V), p[1]) > 1e-4
    m2 = o["accept_len"] >= 2
    assert chi_square_pvalue(np.bincount(o["out_tokens"][m2, 2], minlength=V), p[2]) > 1e-4
    # acceptance rate of the first draft: E[alpha] = sum min(p, q)
    ea = np.minimum(p[0], qs[0].astype(np.float64)).sum()
    n = len(first)
    assert abs(m1.mean() - ea) < 5 * np.sqrt(ea * (1 - ea) / n)
    assert np.all((o["accept_len"] >= 0) & (o["accept_len"] <= 2))
    assert np.all(o["num_out"] == o["accept_len"] + 1)


def test_q_equal_p_always_accepts():
    w, p, qs = _chain_law_case(n=2000, q_mode="equal")
    o = oracle.verify_chain(w)
    assert np.all(o["accept_len"] == 2)


def test_one_hot_q_accepts_with_probability_p():
    V = 6
    x = np.array([[0.0, 1.0, 2.0, 0.5, -1.0, 0.3], [0, 0, 0, 0, 0, 0]], np.float32)
    p = softmax(x[0].astype(np.float64))
    d = 2
    n = 4096
    lg = np.tile(x, (n, 1))
    q = np.zeros((2 * n, V), np.float32)
    q[0::2, d] = 1.0
    q[1::2] = 1.0 / V
    ids = np.tile(np.array([0, d], np.int32), n)
    ua = np.zeros(2 * n, np.float32)
    ua[0::2] = (np.arange(n) / n).astype(np.float32)
    w = chain_workload(lg, "f32", (np.arange(n + 1) * 2), ids, q=q, T=np.ones(n), ua=ua, uf=np.full(n, 0.5))
    o = oracle.verify_chain(w)
    assert abs(o["accept_len"].mean() - p[d]) <= 1.0 / n


# ---------------------------------------------------------------------------
# Trees
# ---------------------------------------------------------------------------


def _all_parent_arrays(N):
    for choice in itertools.product(*[range(i) for i in range(1, N)]):
        yield [-1] + list(choice)


def _brute_force_greedy_path(tokens, parents, argmax_of_node):
    """Longest root path whose every token equals its parent's row argmax and is the
    lowest-index sibling carrying that token; defined over the set of all paths."""
    N = len(tokens)
    best = [0]
    paths = [[0]]
    while paths:
        nxt = []
        for path in paths:
            last = path[-1]
            for c in range(1, N):
                if parents[c] != last:
                    continue
                sib_same = [s for s in range(1, N) if parents[s] == last and tokens[s] == tokens[c]]
                if tokens[c] == argmax_of_node[last] and c == min(sib_same):
                    nxt.append(path + [c])
        for pth in nxt:
            if len(pth) > len(best):
                best = pth
        paths = nxt
    return best


@pytest.mark.parametrize("N", [2, 3, 4, 5, 6])
def test_greedy_tree_brute_force_all_small_trees(N):
    V = 3 if N <= 5 else 2
    rng = np.random.default_rng(100 + N)
    trees = list(_all_parent_arrays(N))
    tok_sets = list(itertools.product(range(V), repeat=N - 1))
    cases = [(t, s) for t in trees for s in tok_sets]
    B = len(cases)
    tokens = np.zeros((B, N), np.int32)
    parents = np.zeros((B, N), np.int32)
    for b, (t, s) in enumerate(cases):
        parents[b] = t
        tokens[b, 0] = 0
        tokens[b, 1:] = s
    lg = rng.integers(0, 3, (B * N, V)).astype(np.float32)  # small integers: ties are frequent
    w = tree_workload(lg, "f32", tokens, parents)
    o = oracle.verify_tree(w, "greedy")
    am = np.argmax(lg, axis=1).reshape(B, N)
    for b in range(B):
        path = _brute_force_greedy_path(tokens[b], parents[b], am[b])
        r = len(path) - 1
        assert o["accept_len"][b] == r
        assert list(o["accept_rows"][b, : r + 1]) == [b * N + i for i in path]
        assert list(o["out_tokens"][b, :r]) == [tokens[b, i] for i in path[1:]]
        assert o["bonus"][b] == am[b, path[-1]]


def test_chain_is_a_tree_special_case():
    w = wl.greedy_chain(batch=40, m=6, vocab=50, dtype="bf16", p_match=0.8, seed=3)
    oc = oracle.verify_chain(w, greedy_all=True)
    L = 7
    tokens = w.verify_ids.reshape(40, L)
    parents = np.tile(np.arange(-1, L - 1, dtype=np.int32), (40, 1))
    ot = oracle.verify_tree(tree_workload(w.logits, "bf16", tokens, parents), "greedy")
    for k in ("accept_len", "num_out", "out_tokens", "bonus", "accept_rows", "commit_cu"):
        assert np.array_equal(oc[k], ot[k]), k


def _target_only_case(n, seed=9, th=1.0, th_single=None, th_acc=None):
    """A fixed small tree, replicated n times with fresh uniforms."""
    rng = np.random.default_rng(seed)
    V, N = 7, 5
    par = np.array([-1, 0, 0, 1, 0], np.int32)  # root children 1,2,4; node 1 has child 3
    tok = np.array([0, 3, 1, 5, 6], np.int32)
    base = (rng.standard_normal((N, V)) * 1.3).astype(np.float32)
    T = 0.8
    lg = np.tile(base, (n, 1))
    w = tree_workload(lg, "f32", np.tile(tok, (n, 1)), np.tile(par, (n, 1)), T=np.full(n, T),
                      ua=wl.uniforms(rng, n * N), uf=wl.uniforms(rng, n), kind="target_only_tree",
                      th_single=th if th_single is None else th_single, th_acc=th if th_acc is None else th_acc)
    p = [softmax(base[i].astype(np.float64) / np.float64(np.float32(T))) for i in range(N)]
    return w, p, tok, par


def test_target_only_tree_output_law():
    n = 60000
    w, p, tok, par = _target_only_case(n)
    o = oracle.verify_tree(w, "target_only", threads=4)
    V = w.vocab
    assert chi_square_pvalue(np.bincount(o["out_tokens"][:, 0], minlength=V), p[0]) > 1e-4
    # after accepting node 1 (token 3) the next token follows node 1's row
    m = (o["accept_len"] >= 1) & (o["out_tokens"][:, 0] == tok[1])
    assert chi_square_pvalue(np.bincount(o["out_tokens"][m, 1], minlength=V), p[1]) > 1e-4
    # accepted child k at the root w.p. p_root(token_k)
    for k in (1, 2, 4):
        frac = np.mean((o["accept_len"] >= 1) & (o["accept_rows"][:, 1] % 5 == k))
        pk = p[0][tok[k]]
        assert abs(frac - pk) < 5 * np.sqrt(pk * (1 - pk) / n) + 1e-9


def test_target_only_children_intervals():
    """At the root the accepted child is the one whose cumulative interval holds u."""
    w, p, tok, par = _target_only_case(1)
    kids = [1, 2, 4]
    c = np.cumsum([p[0][tok[k]] for k in kids])
    edges = [0.0] + list(c)
    for i, k in enumerate(kids):
        for u in (edges[i] + 1e-7, 0.5 * (edges[i] + edges[i + 1]), edges[i + 1] - 1e-7):
            w.u_accept = np.array([u, 0.999, 0.999, 0.999, 0.999], np.float32)
            if abs(np.float64(np.float32(u)) - edges[i + 1]) < 1e-7 or np.float64(np.float32(u)) < edges[i]:
                continue
            o = oracle.verify_tree(w, "target_only")
            assert o["accept_rows"][0, 1] == k
    w.u_accept = np.array([min(0.9999, c[-1] + 1e-4)] + [0.5] * 4, np.float32)
    o = oracle.verify_tree(w, "target_only")
    assert o["accept_len"][0] == 0
    assert o["bonus"][0] not in tok[kids]  # children's tokens are excluded from the stop sample


def test_target_only_with_chain_tree_matches_rejection_of_p():
    """theta = 1 on a chain tree: the emitted sequence follows the target law step by step."""
    n = 40000
    rng = np.random.default_rng(4)
    V, N = 6, 3
    base = (rng.standard_normal((N, V))).astype(np.float32)
    tok = np.array([0, 2, 4], np.int32)
    par = np.array([-1, 0, 1], np.int32)
    w = tree_workload(np.tile(base, (n, 1)), "f32", np.tile(tok, (n, 1)), np.tile(par, (n, 1)),
                      T=np.ones(n), ua=wl.uniforms(rng, n * N), uf=wl.uniforms(rng, n), kind="target_only_tree")
    o = oracle.verify_tree(w, "target_only", threads=4)
    p0 = softmax(base[0].astype(np.float64))
    p1 = softmax(base[1].astype(np.float64))
    assert chi_square_pvalue(np.bincount(o["out_tokens"][:, 0], minlength=V), p0) > 1e-4
    m = o["accept_len"] >= 1
    assert chi_square_pvalue(np.bincount(o["out_tokens"][m, 1], minlength=V), p1) > 1e-4


# Thresholds other than 1 (a lossy rule; these pin the reading written in the
# oracle's header through special cases and the law it implies, with p from
# numpy, not through the oracle's own formula).


def test_target_only_single_threshold_zero_walks_the_first_children():
    """theta_single = 0: every child passes p >= theta_single, so the walk takes the first child at every level
    (root -> node 1 -> node 3, a leaf) whatever the uniforms, and the last token is drawn from the leaf's row."""
    n = 30000
    w, p, tok, par = _target_only_case(n, th_single=0.0, th_acc=1.0)
    o = oracle.verify_tree(w, "target_only", threads=4)
    assert np.all(o["accept_len"] == 2)
    assert np.all(o["out_tokens"][:, 0] == tok[1]) and np.all(o["out_tokens"][:, 1] == tok[3])
    assert np.all(o["accept_rows"][:, :3] % 5 == [0, 1, 3])
    assert chi_square_pvalue(np.bincount(o["out_tokens"][:, 2], minlength=w.vocab), p[3]) > 1e-4


def test_target_only_single_threshold_is_inclusive():
    """p(token) >= theta_single accepts: with theta_single = 0 a first child whose token has probability 0 under
    the root's row (logit -inf) is still accepted."""
    w, p, tok, par = _target_only_case(50, th_single=0.0, th_acc=1.0)
    lg = w.logits.copy()
    lg[0::5, tok[1]] = -np.inf  # every request's root row
    w.logits = lg
    o = oracle.verify_tree(w, "target_only")
    assert np.all(o["accept_len"] >= 1) and np.all(o["accept_rows"][:, 1] % 5 == 1)


def test_target_only_no_child_can_pass_stops_at_the_root():
    """theta_acc huge and theta_single above 1: no child is ever accepted, so every request stops at the root and
    draws from the root's p with the children's tokens removed."""
    n = 30000
    w, p, tok, par = _target_only_case(n, th_single=2.0, th_acc=1e30)
    o = oracle.verify_tree(w, "target_only", threads=4)
    assert np.all(o["accept_len"] == 0)
    q = p[0].copy()
    q[tok[[1, 2, 4]]] = 0.0
    q /= q.sum()
    assert chi_square_pvalue(np.bincount(o["out_tokens"][:, 0], minlength=w.vocab), q) > 1e-4


def test_target_only_single_threshold_picks_the_first_child_above_it():
    """theta_acc huge: only p(token) >= theta_single accepts, so the accepted child is the first one (in sibling
    order) whose probability reaches the threshold, the same for every uniform."""
    w1, p, tok, par = _target_only_case(1)
    kids = [1, 2, 4]
    pk = sorted(p[0][tok[k]] for k in kids)
    for lo, hi in zip(pk[:-1], pk[1:]):
        if hi - lo < 1e-3:
            continue
        th = 0.5 * (lo + hi)
        w, _, _, _ = _target_only_case(200, th_single=th, th_acc=1e30)
        o = oracle.verify_tree(w, "target_only")
        first = next(k for k in kids if p[0][tok[k]] >= th)
        assert np.all(o["accept_len"] >= 1) and np.all(o["accept_rows"][:, 1] % 5 == first)
        if first == 1:  # node 1's only child (node 3) passes iff its probability under node 1's row reaches th
            deeper = p[1][tok[3]] >= th
            assert np.all((o["accept_len"] == 2) == deeper)


def test_target_only_acceptance_threshold_law():
    """theta_single above 1 and theta_acc < 1: at the root child i is accepted w.p.
    min(1, c_i / theta_acc) - min(1, c_(i-1) / theta_acc), c_i the children's cumulative probability in sibling
    order, and the walk stops there w.p. 1 - min(1, c_last / theta_acc)."""
    n = 60000
    th = 0.6
    w, p, tok, par = _target_only_case(n, th_single=2.0, th_acc=th)
    o = oracle.verify_tree(w, "target_only", threads=4)
    kids = [1, 2, 4]
    c = np.cumsum([p[0][tok[k]] for k in kids])
    lo = np.minimum(1.0, np.concatenate([[0.0], c[:-1]]) / th)
    hi = np.minimum(1.0, c / th)
    for k, a, b in zip(kids, lo, hi):
        pk = b - a
        frac = np.mean((o["accept_len"] >= 1) & (o["accept_rows"][:, 1] % 5 == k))
        assert abs(frac - pk) < 5 * np.sqrt(max(pk * (1 - pk), 1e-12) / n) + 1e-9, (k, frac, pk)
    stop = 1.0 - hi[-1]
    assert abs(np.mean(o["accept_len"] == 0) - stop) < 5 * np.sqrt(max(stop * (1 - stop), 1e-12) / n) + 1e-9


def test_empty_residual_falls_back_to_p_and_sets_bit_16():
    """q >= p everywhere on a rejected row leaves [p - q]+ empty: the final token is drawn from p itself (inverse
    CDF over a uniform p of four ids, u = 0.6 -> id 2) and the request reports status bit 16."""
    lg = np.zeros((2, 4), np.float32)                 # p = 1/4 on both rows
    q = np.full((2, 4), 0.5, np.float32)              # not normalised: q(v) > p(v) for every v
    w = chain_workload(lg, "f32", [0, 2], np.array([0, 0], np.int32), q=q, T=np.ones(1),
                       ua=np.array([0.9, 0.5], np.float32), uf=np.array([0.6], np.float32))
    o = oracle.verify_chain(w)
    assert o["accept_len"][0] == 0                    # 0.9 * 0.5 >= 0.25: rejected
    assert int(o["status"][0]) & 16
    assert o["bonus"][0] == 2


def test_repeated_sibling_token_is_skipped_and_flagged():
    """A target-only walk counts a repeated sibling token once and flags it (bit 32): with p = 1/5 everywhere,
    children tokens (3, 3, 1) and u = 0.5 at the root, the cumulative mass reaches 0.2 then 0.4 (not 0.6), no child
    is accepted, and the stop draw over p without ids 3 and 1 takes id 2 for u_final = 0.5."""
    lg = np.zeros((4, 5), np.float32)
    tok = np.array([[0, 3, 3, 1]], np.int32)
    par = np.array([[-1, 0, 0, 0]], np.int32)
    w = tree_workload(lg, "f32", tok, par, T=np.ones(1), ua=np.array([0.5, 0.5, 0.5, 0.5], np.float32),
                      uf=np.array([0.5], np.float32), kind="target_only_tree")
    o = oracle.verify_tree(w, "target_only")
    assert int(o["status"][0]) & 32
    assert o["accept_len"][0] == 0
    assert o["bonus"][0] == 2


def test_nan_in_a_tested_row_is_flagged_and_verification_goes_on():
    """A NaN in a tested row sets status bit 2 and is left out of that row's argmax; the request still accepts the
    row's argmax draft and goes on to its bonus."""
    lg = np.zeros((3, 6), np.float32)
    lg[0, 2], lg[0, 4] = 1.0, np.nan
    lg[1, 1] = 1.0
    lg[2, 5] = 1.0
    w = chain_workload(lg, "f32", [0, 3], np.array([0, 2, 1], np.int32))
    o = oracle.verify_chain(w, greedy_all=True)
    assert o["accept_len"][0] == 2 and o["bonus"][0] == 5
    assert int(o["status"][0]) == 2


def test_target_only_gap_includes_the_single_threshold():
    """With theta_acc huge the cumulative test never decides; when a child's probability sits 1e-9 below
    theta_single the step's gap is that distance, not the uniform's."""
    w, p, tok, par = _target_only_case(1)
    p1 = float(p[0][tok[1]])
    w2, _, _, _ = _target_only_case(1, th_single=p1 + 1e-9, th_acc=1e30)
    o = oracle.verify_tree(w2, "target_only")
    assert o["test_gap"][0, 0] < 1e-8
    assert o["min_gap"][0] < 1e-8


# ---------------------------------------------------------------------------
# Degenerate inputs
# ---------------------------------------------------------------------------


def test_nonfinite_rows_and_bad_layouts():
    V = 8
    lg = np.zeros((6, V), np.float32)
    lg[0, 3] = 2.0
    lg[0, 5] = np.nan
    lg[0, 6] = np.inf  # excluded: argmax stays 3
    lg[1, :] = -np.inf  # unusable row
    lg[2, 1] = 1.0
    ids = np.array([0, 3, 4, 0, 1, 2], np.int32)
    w = chain_workload(lg, "f32", [0, 3, 6], ids)
    o = oracle.verify_chain(w, greedy_all=True)
    assert o["accept_len"][0] == 1 and o["bonus"][0] == -1 and o["status"][0] & 2
    assert o["num_out"][0] == 2
    # bad layouts commit nothing
    w2 = chain_workload(lg, "f32", [0, 4, 3], ids, max_len=6)
    o2 = oracle.verify_chain(w2, greedy_all=True)
    assert o2["status"][1] & 8 and o2["num_out"][1] == 0 and o2["bonus"][1] == -1
    assert o2["commit_cu"][-1] == o2["num_out"][0]
    # a draft id outside [0, V) is a rejection with status bit 1
    ids3 = np.array([0, 99, 4, 0, 1, 2], np.int32)
    o3 = oracle.verify_chain(chain_workload(lg, "f32", [0, 3, 6], ids3), greedy_all=True)
    assert o3["accept_len"][0] == 0 and o3["status"][0] & 1 and o3["bonus"][0] == 3


def test_invalid_tree_verifies_root_only():
    V, N = 5, 4
    lg = np.zeros((N, V), np.float32)
    lg[0, 2] = 1.0
    tok = np.array([[0, 2, 2, 1]], np.int32)
    par = np.array([[-1, 0, 3, 1]], np.int32)  # parent 3 of node 2 is not earlier
    o = oracle.verify_tree(tree_workload(lg, "f32", tok, par), "greedy")
    assert o["status"][0] & 4 and o["accept_len"][0] == 0 and o["bonus"][0] == 2


# ---------------------------------------------------------------------------
# Generator (inputs only)
# ---------------------------------------------------------------------------


def test_bf16_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38], np.float32)
    b = wl.f32_to_bf16_bits(x)
    assert list(b) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x7F62]
    assert np.array_equal(wl.bf16_bits_to_f32(b)[[0, 3]], np.array([1.0, -2.5], np.float32))


def test_generator_is_deterministic_and_shaped():
    a = wl.config(2, vocab=4096)
    b = wl.config(2, vocab=4096)
    assert a.sha256() == b.sha256()
    assert a.logits.shape == (64, 4096) and a.logits.dtype == np.uint16
    assert np.allclose(a.q.sum(axis=1), 1.0, atol=1e-5)
    t = wl.config(3, vocab=2048, batch=2)
    assert t.tokens.shape == (2, 17) and t.parents[0, 0] == -1
    assert np.all(t.parents[:, 1:] < np.arange(1, 17))
    r = wl.config(5, vocab=1024, batch=32)
    lens = np.diff(r.cu_seqlens)
    assert lens.min() >= 1 and lens.max() <= 8 and r.cu_seqlens[-1] == r.rows
