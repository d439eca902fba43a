"""Seeded synthetic inputs for speculative-decoding verification.

This module draws inputs only: target logit rows, anchor and draft tokens,
proposal rows q, caller uniforms, ragged layouts, tree parent arrays, KV slot
ids and sequence lengths.  It contains no part of the verification itself (no
acceptance test, no residual distribution, no inverse-CDF sampling of the
target, no commit bookkeeping).  Both the fp64 oracle and the CUDA path
consume exactly these arrays.

Shapes and value distributions follow the five verification workloads the
pages describe (speculative decoding in SGLang: EAGLE-2 trees, DFlash blocks,
DSpark ragged verify).  Every draw comes from numpy's PCG64 generator with an
explicit seed, so inputs are reproducible on any host.

Proposal-side arithmetic (q = softmax of noised logits; drafting d ~ q) lives
here because it is how a drafter produces its inputs; the verifier only
receives q and d.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

# ----------------------------------------------------------------------------
# bf16 helpers (storage format only)
# ----------------------------------------------------------------------------


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); return raw bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return ((b + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen raw bfloat16 bits to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def uniforms(rng: np.random.Generator, n: int) -> np.ndarray:
    """Uniforms in [0,1) on the grid k * 2^-24, exactly representable in fp32."""
    return (rng.integers(0, 1 << 24, size=n, dtype=np.int64).astype(np.float64) * 2.0 ** -24).astype(np.float32)


# ----------------------------------------------------------------------------
# Workload container
# ----------------------------------------------------------------------------

KINDS = ("greedy_chain", "rejection_chain", "rejection_ragged", "greedy_tree", "target_only_tree",
         "rejection_chain_sparse", "sample_match_chain")


@dataclass
class Workload:
    kind: str
    name: str
    dtype: str                 # "bf16" (uint16 bits) or "f32"
    logits: np.ndarray         # [rows, vocab]
    batch: int
    vocab: int
    rows: int
    max_len: int               # rows per request upper bound (chains: m+1; trees: nodes)
    m: Optional[int] = None    # drafts per request, fixed-length chains
    nodes: Optional[int] = None
    cu_seqlens: Optional[np.ndarray] = None   # int32 [B+1]
    verify_ids: Optional[np.ndarray] = None   # int32 [rows] (row i input token; row i tests verify_ids[i+1])
    q: Optional[np.ndarray] = None            # float32 [rows, vocab]
    cand_ids: Optional[np.ndarray] = None     # int32 [rows, K]: sparse q ids (-1 pads)
    cand_probs: Optional[np.ndarray] = None   # float32 [rows, K]: sparse q probabilities
    temperature: Optional[np.ndarray] = None  # float32 [B]
    u_accept: Optional[np.ndarray] = None     # float32 [rows]
    u_final: Optional[np.ndarray] = None      # float32 [B]
    tokens: Optional[np.ndarray] = None       # int32 [B, nodes]
    parents: Optional[np.ndarray] = None      # int32 [B, nodes]
    first_child: Optional[np.ndarray] = None  # int32 [B, nodes]
    next_sibling: Optional[np.ndarray] = None  # int32 [B, nodes]
    threshold_single: float = 1.0
    threshold_acc: float = 1.0
    row_slots: Optional[np.ndarray] = None    # int64 [rows]
    seq_lens: Optional[np.ndarray] = None     # int64 [B]
    meta: dict = field(default_factory=dict)

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def logit_bytes(self) -> int:
        return self.rows * self.vocab * self.elem_bytes

    def arrays(self) -> dict:
        out = {}
        for k in ("logits", "cu_seqlens", "verify_ids", "q", "cand_ids", "cand_probs", "temperature", "u_accept",
                  "u_final",
                  "tokens", "parents", "first_child", "next_sibling", "row_slots", "seq_lens"):
            v = getattr(self, k)
            if v is not None:
                out[k] = v
        return out

    def sha256(self) -> dict:
        return {k: hashlib.sha256(np.ascontiguousarray(v).tobytes()).hexdigest()[:16]
                for k, v in self.arrays().items()}


# ----------------------------------------------------------------------------
# Drafter-side helpers (inputs to the verifier, not verification)
# ----------------------------------------------------------------------------


def _gaussian_logits(rng: np.random.Generator, rows: int, vocab: int, sigma: float) -> np.ndarray:
    return rng.standard_normal((rows, vocab), dtype=np.float32) * np.float32(sigma)


def _to_storage(x32: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x32) if dtype == "bf16" else np.ascontiguousarray(x32, dtype=np.float32)


def _as_f32(logits: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_f32(logits) if dtype == "bf16" else logits


def _proposal_rows(rng: np.random.Generator, target32: np.ndarray, scale: np.ndarray,
                   noise_sigma: float, chunk: int = 64) -> np.ndarray:
    """q_row = softmax(target_row * scale_row + noise_sigma * N(0,1)), normalised in fp64.

    This is how the synthetic drafter forms its proposal; `scale` is 1/T for a
    drafter that matches the target's temperature.
    """
    rows, vocab = target32.shape
    q = np.empty((rows, vocab), dtype=np.float32)
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        z = target32[r0:r1].astype(np.float64) * scale[r0:r1, None]
        z += noise_sigma * rng.standard_normal((r1 - r0, vocab), dtype=np.float32)
        z -= z.max(axis=1, keepdims=True)
        np.exp(z, out=z)
        z /= z.sum(axis=1, keepdims=True)
        q[r0:r1] = z
    return q


def _draw_from_rows(rng: np.random.Generator, q: np.ndarray) -> np.ndarray:
    """Draft tokens d ~ q_row by inverse CDF with the drafter's own uniforms."""
    rows, vocab = q.shape
    u = rng.random(rows)
    out = np.empty(rows, dtype=np.int32)
    for i in range(rows):
        c = np.cumsum(q[i], dtype=np.float64)
        out[i] = min(int(np.searchsorted(c, u[i] * c[-1], side="right")), vocab - 1)
    return out


# ----------------------------------------------------------------------------
# Chains (fixed m) and ragged blocks
# ----------------------------------------------------------------------------


def greedy_chain(batch: int = 1, m: int = 4, vocab: int = 32000, dtype: str = "f32", sigma: float = 3.0,
                 p_match: float = 0.7, seed: int = 1001, name: str = "greedy_chain") -> Workload:
    """Greedy chain verify: each draft equals its row's argmax w.p. p_match, else a uniform id.

    Logits i.i.d. N(0, sigma^2).  Rows are row-aligned: row i's input token is
    verify_ids[i] (the anchor at each request's first row).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    L = m + 1
    R = batch * L
    x = _gaussian_logits(rng, R, vocab, sigma)
    logits = _to_storage(x, dtype)
    xv = _as_f32(logits, dtype)
    ids = rng.integers(0, vocab, size=R, dtype=np.int64).astype(np.int32)
    for b in range(batch):
        for j in range(m):
            row = b * L + j
            if rng.random() < p_match:
                ids[row + 1] = int(np.argmax(xv[row]))
    cu = (np.arange(batch + 1, dtype=np.int64) * L).astype(np.int32)
    return Workload(kind="greedy_chain", name=name, dtype=dtype, logits=logits, batch=batch, vocab=vocab,
                    rows=R, max_len=L, m=m, cu_seqlens=cu, verify_ids=ids,
                    row_slots=rng.permutation(1 << 20)[:R].astype(np.int64),
                    seq_lens=rng.integers(128, 4097, size=batch).astype(np.int64),
                    meta={"seed": seed, "sigma": sigma, "p_match": p_match})


def rejection_chain(batch: int = 8, m: int = 7, vocab: int = 151936, dtype: str = "bf16", sigma: float = 3.0,
                    boost: float = 6.0, temperature: float = 0.8, noise_sigma: float = 1.0,
                    drafter_uses_temperature: bool = True, seed: int = 1002,
                    name: str = "rejection_chain", kind: str = "rejection_chain") -> Workload:
    """p/q rejection chain: fixed m drafts per request, q from noised target softmax, d ~ q.

    boost > 0 adds +boost to one uniformly chosen id per row before rounding.
    drafter_uses_temperature: q = softmax(l/T + noise) if True, else softmax(l + noise).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    L = m + 1
    R = batch * L
    x = _gaussian_logits(rng, R, vocab, sigma)
    if boost:
        hot = rng.integers(0, vocab, size=R)
        x[np.arange(R), hot] += np.float32(boost)
    logits = _to_storage(x, dtype)
    xv = _as_f32(logits, dtype)
    T = np.full(batch, temperature, dtype=np.float32)
    scale = np.full(R, 1.0 / float(np.float32(temperature)) if drafter_uses_temperature else 1.0)
    q = _proposal_rows(rng, xv, scale, noise_sigma)
    d = _draw_from_rows(rng, q)
    ids = rng.integers(0, vocab, size=R, dtype=np.int64).astype(np.int32)
    for b in range(batch):
        for j in range(m):
            ids[b * L + j + 1] = d[b * L + j]
    cu = (np.arange(batch + 1, dtype=np.int64) * L).astype(np.int32)
    return Workload(kind=kind, name=name, dtype=dtype, logits=logits, batch=batch, vocab=vocab, rows=R,
                    max_len=L, m=m, cu_seqlens=cu, verify_ids=ids, q=q, temperature=T,
                    u_accept=uniforms(rng, R), u_final=uniforms(rng, batch),
                    row_slots=rng.permutation(1 << 20)[:R].astype(np.int64),
                    seq_lens=rng.integers(128, 4097, size=batch).astype(np.int64),
                    meta={"seed": seed, "sigma": sigma, "boost": boost, "T": temperature,
                          "noise_sigma": noise_sigma})


def rejection_chain_sparse(batch: int = 8, m: int = 7, vocab: int = 151936, dtype: str = "bf16", K: int = 16,
                           sigma: float = 3.0, boost: float = 6.0, temperature: float = 0.8, noise_sigma: float = 1.0,
                           pad: int = 0, seed: int = 1006, name: str = "rejection_chain_sparse") -> Workload:
    """p/q rejection chain whose q has K nonzeros (a candidate selector, [E2D] §6.2, §6.5).

    Per row the drafter scores every id with l/T + noise, keeps the K best as
    candidates (score order), sets q = softmax over the candidates' scores and
    draws the draft by inverse CDF over the candidates in that order.  `pad`
    trailing entries per row carry id -1 (padding) with a nonzero probability
    that must be ignored.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    L = m + 1
    R = batch * L
    x = _gaussian_logits(rng, R, vocab, sigma)
    if boost:
        hot = rng.integers(0, vocab, size=R)
        x[np.arange(R), hot] += np.float32(boost)
    logits = _to_storage(x, dtype)
    xv = _as_f32(logits, dtype)
    T = np.full(batch, temperature, dtype=np.float32)
    Kc = min(K, vocab)
    cand = np.full((R, Kc + pad), -1, dtype=np.int32)
    prob = np.zeros((R, Kc + pad), dtype=np.float32)
    d = np.empty(R, dtype=np.int32)
    u = rng.random(R)
    for r in range(R):
        z = xv[r].astype(np.float64) / float(np.float32(temperature))
        z += noise_sigma * rng.standard_normal(vocab)
        top = np.argpartition(-z, Kc - 1)[:Kc]
        top = top[np.argsort(-z[top], kind="stable")]
        e = np.exp(z[top] - z[top].max())
        pr = e / e.sum()
        cand[r, :Kc] = top
        prob[r, :Kc] = pr
        prob[r, Kc:] = 0.5
        c = np.cumsum(pr)
        d[r] = top[min(int(np.searchsorted(c, u[r] * c[-1], side="right")), Kc - 1)]
    ids = rng.integers(0, vocab, size=R, dtype=np.int64).astype(np.int32)
    for b in range(batch):
        for j in range(m):
            ids[b * L + j + 1] = d[b * L + j]
    cu = (np.arange(batch + 1, dtype=np.int64) * L).astype(np.int32)
    return Workload(kind="rejection_chain_sparse", name=name, dtype=dtype, logits=logits, batch=batch,
                    vocab=vocab, rows=R, max_len=L, m=m, cu_seqlens=cu, verify_ids=ids, cand_ids=cand,
                    cand_probs=prob, temperature=T, u_accept=uniforms(rng, R), u_final=uniforms(rng, batch),
                    row_slots=rng.permutation(1 << 20)[:R].astype(np.int64),
                    seq_lens=rng.integers(128, 4097, size=batch).astype(np.int64),
                    meta={"seed": seed, "sigma": sigma, "boost": boost, "T": temperature, "K": K,
                          "noise_sigma": noise_sigma, "pad": pad})


def ragged_block(batch: int = 256, max_len: int = 8, vocab: int = 151936, dtype: str = "bf16",
                 sigma: float = 3.0, t_lo: float = 0.5, t_hi: float = 1.2, noise_sigma: float = 1.0,
                 lens: Optional[list] = None, seed: int = 1005, name: str = "rejection_ragged") -> Workload:
    """DSpark-style ragged verify: per-request verify length (anchor included) uniform in 1..max_len.

    Temperature per request U(t_lo, t_hi); q = softmax(l/T_b + noise); KV slots are
    a random permutation of a 2^20-slot pool; seq_lens U{128..4096}.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    if lens is None:
        lens = rng.integers(1, max_len + 1, size=batch)
    lens = np.asarray(lens, dtype=np.int64)
    batch = len(lens)
    cu = np.zeros(batch + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lens)
    R = int(cu[-1])
    x = _gaussian_logits(rng, R, vocab, sigma)
    logits = _to_storage(x, dtype)
    xv = _as_f32(logits, dtype)
    T = rng.uniform(t_lo, t_hi, size=batch).astype(np.float32)
    row_req = np.repeat(np.arange(batch), lens)
    scale = 1.0 / T.astype(np.float64)[row_req]
    q = _proposal_rows(rng, xv, scale, noise_sigma)
    d = _draw_from_rows(rng, q)
    ids = rng.integers(0, vocab, size=R, dtype=np.int64).astype(np.int32)
    for b in range(batch):
        for j in range(int(lens[b]) - 1):
            ids[cu[b] + j + 1] = d[cu[b] + j]
    return Workload(kind="rejection_ragged", name=name, dtype=dtype, logits=logits, batch=batch, vocab=vocab,
                    rows=R, max_len=int(max_len), cu_seqlens=cu.astype(np.int32), verify_ids=ids, q=q,
                    temperature=T, u_accept=uniforms(rng, R), u_final=uniforms(rng, batch),
                    row_slots=rng.permutation(1 << 20)[:R].astype(np.int64),
                    seq_lens=rng.integers(128, 4097, size=batch).astype(np.int64),
                    meta={"seed": seed, "sigma": sigma, "T_range": (t_lo, t_hi), "noise_sigma": noise_sigma})


# ----------------------------------------------------------------------------
# EAGLE-2 style trees
# ----------------------------------------------------------------------------


def eagle2_tree(batch: int = 16, topk: int = 4, depth: int = 5, keep: int = 16, vocab: int = 128256,
                dtype: str = "bf16", sigma: float = 3.0, noise_sigma: float = 1.0, temperature: float = 1.0,
                mode: str = "greedy_tree", seed: int = 1003, name: Optional[str] = None) -> Workload:
    """EAGLE-2 dynamic tree (expand / rerank with path-product scores), one target row per node.

    Every candidate c carries its own target row L_c ~ N(0, sigma^2) (a pure
    function of seed, request and generation index).  The drafter at an
    expanded node c proposes q_c = softmax(L_c + noise); its top-k tokens become
    c's children with score = score(c) * q_c(token).  Per depth the frontier
    keeps the top-k of the k^2 new candidates; at the end all candidates are
    reranked and the top `keep` kept.  Ties: depth ascending, then generation
    index.  Node order: root, then (depth asc, score desc, generation asc).
    """
    assert mode in ("greedy_tree", "target_only_tree")
    rng = np.random.Generator(np.random.PCG64(seed))
    N = keep + 1
    lg = np.empty((batch * N, vocab), dtype=np.uint16 if dtype == "bf16" else np.float32)
    tokens = np.empty((batch, N), dtype=np.int32)
    parents = np.empty((batch, N), dtype=np.int32)

    def node_row(b, g):
        r = np.random.Generator(np.random.PCG64([seed, b, g]))
        return _to_storage(r.standard_normal(vocab, dtype=np.float32) * np.float32(sigma), dtype)

    for b in range(batch):
        nrng = np.random.Generator(np.random.PCG64([seed, b, 1 << 30]))
        # candidate table: gen index -> (depth, score, token, parent gen)
        cand = {0: (0, 1.0, int(rng.integers(0, vocab)), -1)}
        rows_cache = {}
        next_gen = 1
        frontier = [0]
        all_cands = []
        for dpt in range(1, depth + 1):
            new = []
            for g in frontier:
                if g not in rows_cache:
                    rows_cache[g] = node_row(b, g)
                z = _as_f32(rows_cache[g][None, :], dtype)[0].astype(np.float64)
                z = z + noise_sigma * nrng.standard_normal(vocab)
                z -= z.max()
                e = np.exp(z)
                qv = e / e.sum()
                top = np.argsort(-qv, kind="stable")[:topk]
                for t in top:
                    sc = float(np.float32(np.float32(cand[g][1]) * np.float32(qv[t])))
                    cand[next_gen] = (dpt, sc, int(t), g)
                    new.append(next_gen)
                    next_gen += 1
            all_cands.extend(new)
            new.sort(key=lambda gg: (-cand[gg][1], cand[gg][0], gg))
            frontier = new[:topk]
        all_cands.sort(key=lambda gg: (-cand[gg][1], cand[gg][0], gg))
        kept = set(all_cands[:keep])
        for gg in kept:  # ancestor closure holds for monotone scores with this tie rule
            p = cand[gg][3]
            assert p == 0 or p in kept
        order = [0] + sorted(kept, key=lambda gg: (cand[gg][0], -cand[gg][1], gg))
        pos = {g: i for i, g in enumerate(order)}
        for i, g in enumerate(order):
            tokens[b, i] = cand[g][2]
            parents[b, i] = -1 if i == 0 else pos[cand[g][3]]
            if g not in rows_cache:
                rows_cache[g] = node_row(b, g)
            lg[b * N + i] = rows_cache[g]
    R = batch * N
    w = Workload(kind=mode, name=name or mode, dtype=dtype, logits=lg, batch=batch, vocab=vocab, rows=R,
                 max_len=N, nodes=N, tokens=tokens, parents=parents,
                 row_slots=rng.permutation(1 << 20)[:R].astype(np.int64),
                 seq_lens=rng.integers(128, 4097, size=batch).astype(np.int64),
                 meta={"seed": seed, "topk": topk, "depth": depth, "keep": keep, "sigma": sigma,
                       "noise_sigma": noise_sigma})
    if mode == "target_only_tree":
        w.temperature = np.full(batch, temperature, dtype=np.float32)
        w.u_accept = uniforms(rng, R)
        w.u_final = uniforms(rng, batch)
    return w


def sibling_lists(parents: np.ndarray) -> tuple:
    """first_child / next_sibling arrays that list each node's children in ascending index."""
    B, N = parents.shape
    fc = np.full((B, N), -1, dtype=np.int32)
    ns = np.full((B, N), -1, dtype=np.int32)
    for b in range(B):
        last = {}
        for i in range(1, N):
            p = int(parents[b, i])
            if p in last:
                ns[b, last[p]] = i
            else:
                fc[b, p] = i
            last[p] = i
    return fc, ns


# ----------------------------------------------------------------------------
# The five named workloads
# ----------------------------------------------------------------------------


def config(index: int, **overrides) -> Workload:
    """The five verification workloads, seeded with 1000 + index.

    1 greedy chain, B=1, m=4, V=32000, fp32
    2 rejection chain, B=8, m=7, V=151936, bf16, +6 boost, T=0.8
    3 EAGLE-2 tree, B=16, topk 4, depth 5, 16 drafts + root, V=128256, bf16
      (mode greedy_tree or target_only_tree via overrides)
    4 DFlash block, B=64, anchor + 15, V=151936, bf16, q noise 1.5, T=1
    5 DSpark ragged, B=256, lens U{1..8}, V=151936, bf16, T U(0.5,1.2)
    """
    seed = 1000 + index
    if index == 1:
        kw = dict(batch=1, m=4, vocab=32000, dtype="f32", seed=seed, name="c1_greedy_chain")
        kw.update(overrides)
        return greedy_chain(**kw)
    if index == 2:
        kw = dict(batch=8, m=7, vocab=151936, dtype="bf16", boost=6.0, temperature=0.8, noise_sigma=1.0,
                  drafter_uses_temperature=True, seed=seed, name="c2_rejection_chain")
        kw.update(overrides)
        return rejection_chain(**kw)
    if index == 3:
        kw = dict(batch=16, topk=4, depth=5, keep=16, vocab=128256, dtype="bf16", mode="greedy_tree",
                  seed=seed)
        kw.update(overrides)
        kw.setdefault("name", "c3_" + kw["mode"])
        return eagle2_tree(**kw)
    if index == 4:
        kw = dict(batch=64, m=15, vocab=151936, dtype="bf16", boost=0.0, temperature=1.0, noise_sigma=1.5,
                  drafter_uses_temperature=False, seed=seed, name="c4_dflash_block")
        kw.update(overrides)
        return rejection_chain(**kw)
    if index == 5:
        kw = dict(batch=256, max_len=8, vocab=151936, dtype="bf16", seed=seed, name="c5_dspark_ragged")
        kw.update(overrides)
        return ragged_block(**kw)
    raise ValueError(index)


# ----------------------------------------------------------------------------
# Inputs of the verify-length scheduler and of the tree-input builder
# ----------------------------------------------------------------------------


def dspark_schedule(requests: int = 256, drafts: int = 15, seed: int = 1006) -> dict:
    """Survival scores of a DSpark-style block ([E2D] §5.6.3–5.6.4): per request, the running product of
    per-position confidences drawn U(0.5, 1); the previous round's survivals stand in for the history; the speed
    table (rounds/s by target rows M) falls as 1 / (1 + M / 500)."""
    rng = np.random.default_rng(seed)
    conf = rng.uniform(0.5, 1.0, size=(requests, drafts)).astype(np.float32)
    survival = np.cumprod(conf, axis=1, dtype=np.float32)
    hist = np.cumprod(rng.uniform(0.5, 1.0, size=(requests, drafts)).astype(np.float32), axis=1,
                      dtype=np.float32).ravel()
    sps = (1.0 / (1.0 + np.arange(requests * (drafts + 1) + 1) / 500.0)).astype(np.float32)
    return {"survival": survival, "hist": hist, "sps": sps}


def random_trees(batch: int = 64, nodes: int = 64, fan: int = 8, seed: int = 1007) -> dict:
    """Parent arrays of draft trees: node i's parent is uniform among the fan nodes before it (chains when
    fan = 1, bushy trees otherwise), the root first; sequence lengths U{128..4096}."""
    rng = np.random.default_rng(seed)
    parents = np.empty((batch, nodes), np.int32)
    parents[:, 0] = -1
    for i in range(1, nodes):
        parents[:, i] = rng.integers(max(0, i - fan), i, size=batch)
    seq_lens = rng.integers(128, 4097, size=batch).astype(np.int64)
    return {"parents": parents, "seq_lens": seq_lens}
