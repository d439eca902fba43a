"""CUDA path vs the fp64 oracle, element by element, on the same seeded inputs.

Token decisions (argmax, accepted lengths, token ids, commit indices, status
bits) must be bit-exact on every request whose decisions are not within 1e-6
of a threshold (those are counted and reported).  Probabilities must agree to
1e-5 absolute for fp32 logits and 2e-3 for bf16 logits; the tests also hold
the row normaliser Z to 2e-6 relative.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from reject_row_vocab_gb300 import _build  # noqa: E402
from reject_row_vocab_gb300 import workload as wl  # noqa: E402
from tests.gpu_compare import compare, flag_bound, oracle_outputs  # noqa: E402
from tests.helpers import chain_workload, tree_workload  # noqa: E402

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

_build.build()
from reject_row_vocab_gb300 import device_workload as dw  # noqa: E402
from reject_row_vocab_gb300 import specverify as sv  # noqa: E402

def run_gpu(w, use_lists=False, ws=None, out=None):
    d = dw.DeviceInputs.from_workload(w)
    if ws is None:
        ws = dw.workspace_for(w)
    o = dw.run(w, d, out=out, ws=ws, use_lists=use_lists)
    torch.cuda.synchronize()
    return o.to_numpy()


def check(w, use_lists=False):
    g = run_gpu(w, use_lists=use_lists)
    o = oracle_outputs(w, use_lists=use_lists)
    res = compare(w, g, o)
    return g, o, res


# ---------------------------------------------------------------------------
# Row statistics and probabilities
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,V", [(4, 1), (5, 3), (3, 7), (9, 16), (7, 1000), (33, 4099), (2, 151936),
                                    (3000, 64), (5, 32000),
                                    (40, 262147)])  # 33 (bf16) or 64 (fp32) one-stage chunks per tail row
def test_row_stats_and_probabilities(dtype, rows, V):
    rng = np.random.default_rng(rows * 1000 + V)
    x = (rng.standard_normal((rows, V)) * 3).astype(np.float32)
    if V > 4:
        x[0, V // 2] = x[0, V // 3] = x[0].max() + 1.0  # tie: lowest index
    logits = wl.f32_to_bf16_bits(x) if dtype == "bf16" else x
    T = rng.uniform(0.4, 1.6, rows).astype(np.float32)
    T[::5] = 0.0  # greedy rows
    probe = rng.integers(0, V, rows).astype(np.int32)
    probe[1 % rows] = np.argmax(wl.bf16_bits_to_f32(logits[1 % rows]) if dtype == "bf16" else x[1 % rows])
    ref = oracle.row_stats(logits, dtype, row_temp=T, probe=probe)
    t = dw.padded_rows(dw._to_tensor(logits), "cuda")
    r = sv.row_stats(t, row_temp=torch.from_numpy(T).cuda(), probe=torch.from_numpy(probe).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(r["argmax"].cpu().numpy(), ref["argmax"])
    assert np.array_equal(r["max"].cpu().numpy().astype(np.float64), ref["max"])
    z = r["z"].cpu().numpy()
    samp = T > 0
    assert np.all(z[~samp] == 0)
    assert np.all(np.abs(z[samp] - ref["z"][samp]) <= 2e-6 * ref["z"][samp])
    p = r["p"].cpu().numpy().astype(np.float64)
    tol = 1e-5 if dtype == "f32" else 2e-3
    assert np.all(np.abs(p - ref["p"]) <= tol)
    assert np.all(np.abs(p - ref["p"]) <= 2e-6 * np.maximum(ref["p"], 1e-30) + 1e-12)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("with_probe", [False, True])
@pytest.mark.parametrize("V", [4099, 151936])
def test_row_stats_extreme_temperatures(dtype, with_probe, V):
    # Low temperatures move the exponent reference often (the bound sits 16/k logits above it), high ones never;
    # wide rows make l*k large.  Z must stay within 2e-6 of the fp64 oracle, max and argmax exact.
    rng = np.random.default_rng(V + (7 if with_probe else 0) + (1 if dtype == "bf16" else 0))
    temps = [0.01, 0.05, 0.25, 0.5, 1.0, 4.0, 100.0]
    rows = 2 * len(temps) + 2
    x = (rng.standard_normal((rows, V)) * 3).astype(np.float32)
    x[len(temps):2 * len(temps)] *= 20.0  # wide rows: logits up to about +-250
    x[-2] = 1.5  # all equal: Z = V exactly
    x[-1] = -np.inf
    x[-1, V // 3] = 2.0  # a single usable entry: Z = 1
    logits = wl.f32_to_bf16_bits(x) if dtype == "bf16" else x
    T = np.array(temps * 2 + [0.3, 0.3], dtype=np.float32)
    probe = rng.integers(0, V, rows).astype(np.int32) if with_probe else None
    ref = oracle.row_stats(logits, dtype, row_temp=T, probe=probe)
    t = dw.padded_rows(dw._to_tensor(logits), "cuda")
    r = sv.row_stats(t, row_temp=torch.from_numpy(T).cuda(),
                     probe=torch.from_numpy(probe).cuda() if with_probe else None)
    torch.cuda.synchronize()
    assert np.array_equal(r["argmax"].cpu().numpy(), ref["argmax"])
    assert np.array_equal(r["max"].cpu().numpy().astype(np.float64), ref["max"])
    z = r["z"].cpu().numpy()
    assert np.all(np.abs(z - ref["z"]) <= 2e-6 * ref["z"]), np.max(np.abs(z - ref["z"]) / ref["z"])
    assert z[-2] == V and z[-1] == 1.0
    if with_probe:
        p = r["p"].cpu().numpy().astype(np.float64)
        assert np.all(np.abs(p - ref["p"]) <= 2e-6 * np.maximum(ref["p"], 1e-30) + 1e-12)


# ---------------------------------------------------------------------------
# Small cases spanning several tiles and a ragged tail
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [1, 2, 3, 7, 16, 1000, 4099, 32000])
def test_greedy_chain_small(dtype, V):
    w = wl.greedy_chain(batch=6, m=5, vocab=V, dtype=dtype, p_match=0.8, seed=V)
    check(w)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [2, 7, 16, 1000, 4099, 20011])
def test_rejection_chain_small(dtype, V):
    w = wl.rejection_chain(batch=9, m=6, vocab=V, dtype=dtype, boost=2.0, temperature=0.9, noise_sigma=0.7,
                           seed=V + 1)
    check(w)


@pytest.mark.parametrize("V", [3, 999, 7777])
def test_ragged_small(V):
    w = wl.ragged_block(batch=40, max_len=8, vocab=V, seed=V + 2)
    check(w)
    w1 = wl.ragged_block(lens=[1, 1, 3, 1, 8], max_len=8, vocab=V, seed=V + 3)  # bonus-only requests
    check(w1)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rejection_chain_more_than_32_chunks_per_row(dtype):
    # V = 262147: tail rows hold 33 (bf16) or 64 (fp32) chunks, so the row merge's lanes fold several each
    w = wl.rejection_chain(batch=8, m=7, vocab=262147, dtype=dtype, seed=262 + (dtype == "bf16"),
                           name="chain_v262147_" + dtype)
    check(w)


@pytest.mark.parametrize("batch", [511, 512, 2000])
def test_ragged_batch_around_the_staged_table_size(batch):
    # Up to 511 requests the statistics kernel stages the request offsets (batch + 1 entries) and temperatures in
    # shared memory; beyond, each chunk's row finds its request by searching cu_seqlens in global memory.
    w = wl.ragged_block(batch=batch, max_len=8, vocab=4099, seed=batch + 5)
    g, o, res = check(w)
    assert res["requests"] == batch


@pytest.mark.parametrize("mode", ["greedy_tree", "target_only_tree"])
@pytest.mark.parametrize("batch,topk,depth,keep", [(4, 16, 16, 256), (12, 16, 16, 256), (6, 8, 16, 128),
                                                   (2, 32, 40, 1023)])  # the last: the 1024-node maximum
def test_tree_large(mode, batch, topk, depth, keep):
    # 129 and 257 nodes per request; greedy batches whose node arrays fit the one-CTA accept-and-commit kernel
    # (4 x 257 nodes) and batches that do not (12 x 257 nodes) take different kernels.
    w = wl.eagle2_tree(batch=batch, topk=topk, depth=depth, keep=keep, vocab=2048, mode=mode, noise_sigma=0.5,
                       seed=batch * 100 + keep, name="tree_large_%s_%d" % (mode, keep + 1))
    check(w)


@pytest.mark.parametrize("mode", ["greedy_tree", "target_only_tree"])
@pytest.mark.parametrize("V,keep", [(64, 6), (2000, 16), (5003, 30)])
def test_tree_small(mode, V, keep):
    w = wl.eagle2_tree(batch=12, topk=3, depth=4, keep=keep, vocab=V, mode=mode, noise_sigma=0.5,
                       temperature=0.9, seed=V + keep)
    check(w)
    w.first_child, w.next_sibling = wl.sibling_lists(w.parents)
    check(w, use_lists=True)


@pytest.mark.parametrize("th_single,th_acc", [(0.0, 1.0), (2.0, 1e30), (0.3, 0.7), (0.05, 0.5), (1.5, 0.25)])
def test_target_only_thresholds(th_single, th_acc):
    """Target-only walks with thresholds other than 1 (first child always; never a child; single-token and
    cumulative acceptance mixed) match the oracle, with and without sibling lists."""
    import dataclasses
    w = wl.eagle2_tree(batch=10, topk=4, depth=4, keep=20, vocab=4099, mode="target_only_tree", noise_sigma=0.5,
                       temperature=0.9, seed=int(th_single * 100 + th_acc * 10) % 1000 + 3)
    w = dataclasses.replace(w, threshold_single=th_single, threshold_acc=th_acc)
    check(w)
    w.first_child, w.next_sibling = wl.sibling_lists(w.parents)
    check(w, use_lists=True)


@pytest.mark.parametrize("batch", [1, 32, 33, 70])
def test_greedy_batch_sizes_around_the_single_cta_path(batch):
    """Greedy calls of at most 32 requests are accepted and committed by one CTA; larger ones by the acceptance
    and commit kernels: both match the oracle."""
    check(wl.greedy_chain(batch=batch, m=5, vocab=3001, dtype="bf16", p_match=0.8, seed=batch))
    w = wl.eagle2_tree(batch=batch, topk=3, depth=3, keep=8, vocab=2048, mode="greedy_tree", seed=batch + 1)
    check(w)
    w.first_child, w.next_sibling = wl.sibling_lists(w.parents)
    check(w, use_lists=True)


@pytest.mark.parametrize("batch,m", [(16, 63), (20, 63)])
def test_single_cta_commit_with_slots_staged_or_read(batch, m):
    """The one-CTA greedy path copies the KV slots of up to 1024 rows to shared memory before its wait (16 x 64
    rows) and reads them from global memory beyond that (20 x 64 rows): the commit lists match the oracle."""
    check(wl.greedy_chain(batch=batch, m=m, vocab=3001, dtype="bf16", p_match=0.93, seed=batch + m))


def test_chain_and_tree_entry_points_agree():
    w = wl.greedy_chain(batch=20, m=7, vocab=3000, dtype="bf16", p_match=0.85, seed=5)
    L = 8
    t = tree_workload(w.logits, "bf16", w.verify_ids.reshape(20, L), np.tile(np.arange(-1, L - 1), (20, 1)))
    g1 = run_gpu(w)
    g2 = run_gpu(t)
    for k in ("accept_len", "num_out", "out_tokens", "bonus", "accept_rows", "commit_cu"):
        assert np.array_equal(g1[k], g2[k]), k


# ---------------------------------------------------------------------------
# The five workloads at full size (the launch configuration the benchmark times)
# ---------------------------------------------------------------------------


@pytest.mark.parametrize("idx,mode", [(1, None), (2, None), (3, "greedy_tree"), (3, "target_only_tree"), (4, None),
                                      (5, None)])
def test_full_size_configs(idx, mode):
    w = wl.config(idx, mode=mode) if mode else wl.config(idx)
    g, o, res = check(w)
    # A request is flagged when a decision's uniform lies within 1e-6 of its threshold; over a
    # 152k-entry vocabulary about 3 % of draws land on a token whose whole CDF interval is that
    # narrow.  Flagged requests are still compared up to that decision; the counts are bounded.
    msg = "%s: %d requests, %d exact, %d draw-flagged, %d test-flagged, %d differ" % (
        w.name, res["requests"], res["exact"], res["draw_flagged"], res["test_flagged"], res["differ"])
    assert res["draw_flagged"] <= flag_bound(w.batch, 0.15), msg
    assert res["test_flagged"] <= flag_bound(w.batch, 0.05), msg
    assert res["differ"] <= res["flagged"], msg
    # accepted lengths stay within [0, max_len - 1]; tau = E[r + 1] within [1, k + 1]
    assert np.all((g["accept_len"] >= 0) & (g["accept_len"] < w.max_len))


# ---------------------------------------------------------------------------
# Degenerate inputs
# ---------------------------------------------------------------------------


def test_nonfinite_and_unusable_rows():
    V = 300
    rng = np.random.default_rng(1)
    x = rng.standard_normal((8, V)).astype(np.float32)
    x[0, 5] = np.nan
    x[0, 9] = np.inf
    x[1, :] = -np.inf
    x[4, 100] = -np.inf
    x[5, :] = -np.inf
    x[5, 17] = np.nan
    ids = rng.integers(0, V, 8).astype(np.int32)
    ids[1] = int(np.nanargmax(np.where(np.isfinite(x[0]), x[0], -np.inf)))
    for dtype in ("f32", "bf16"):
        lg = wl.f32_to_bf16_bits(x) if dtype == "bf16" else x
        check(chain_workload(lg, dtype, [0, 4, 8], ids, name="nonfinite_" + dtype))
        q = np.full((8, V), 1.0 / V, np.float32)
        check(chain_workload(lg, dtype, [0, 4, 8], ids, q=q, T=[1.0, 0.7], ua=np.full(8, 0.3), uf=[0.2, 0.9],
                             name="nonfinite_rej_" + dtype))


def test_bad_layouts_and_token_ranges():
    V = 500
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((12, V)) * 2).astype(np.float32)
    ids = rng.integers(0, V, 12).astype(np.int32)
    ids[1] = -5
    ids[7] = V + 3
    q = np.full((12, V), 1.0 / V, np.float32)
    for cu in ([0, 3, 2, 12], [0, 4, 8, 13], [0, 12, 12, 12], [0, 1, 2, 3]):
        w = chain_workload(x, "f32", cu, ids, q=q, T=[1.0, 1.0, 0.0], ua=np.full(12, 0.5), uf=[0.1, 0.5, 0.9],
                           max_len=6, name="bad_cu")
        check(w)


def test_empty_batch():
    d = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    o = sv.greedy_chain(d, torch.zeros(0, dtype=torch.int32, device="cuda"), 3)
    torch.cuda.synchronize()
    assert o.commit_cu.cpu().tolist() == [0]


def test_single_row_requests_and_m_zero():
    w = wl.rejection_chain(batch=17, m=0, vocab=3001, dtype="bf16", seed=8)
    g, o, _ = check(w)
    assert np.all(g["accept_len"] == 0) and np.all(g["num_out"] == 1)
    check(wl.greedy_chain(batch=5, m=0, vocab=100, dtype="f32", seed=9))


def test_q_equal_p_accepts_everything():
    V = 700
    rng = np.random.default_rng(4)
    B, L = 10, 5
    x = (rng.standard_normal((B * L, V)) * 2).astype(np.float32)
    T = 0.8
    p = np.exp((x - x.max(1, keepdims=True)) / np.float32(T))
    p /= p.sum(1, keepdims=True)
    ids = rng.integers(0, V, B * L).astype(np.int32)
    w = chain_workload(x, "f32", np.arange(B + 1) * L, ids, q=p.astype(np.float32), T=np.full(B, T),
                       ua=np.minimum(wl.uniforms(rng, B * L), 0.999), uf=wl.uniforms(rng, B))
    g, o, _ = check(w)
    assert np.all(g["accept_len"] == L - 1)


def test_invalid_trees_and_duplicate_siblings():
    V, N, B = 50, 6, 4
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((B * N, V)) * 2).astype(np.float32)
    par = np.tile(np.array([-1, 0, 0, 1, 1, 2], np.int32), (B, 1))
    tok = rng.integers(0, V, (B, N)).astype(np.int32)
    par[1, 3] = 4  # forward parent: invalid
    par[2, 0] = 0  # root with a parent: invalid
    tok[3, 2] = tok[3, 1]  # duplicate siblings
    tok[0, 1] = int(np.argmax(x[0]))
    tok[3, 1] = int(np.argmax(x[3 * N]))
    tok[3, 2] = tok[3, 1]
    for kind in ("greedy_tree", "target_only_tree"):
        w = tree_workload(x, "f32", tok, par, T=np.full(B, 0.9), ua=wl.uniforms(rng, B * N), uf=wl.uniforms(rng, B),
                          kind=kind)
        check(w)


def test_workspace_reuse_gives_identical_results():
    w = wl.ragged_block(batch=64, max_len=8, vocab=5000, seed=11)
    d = dw.DeviceInputs.from_workload(w)
    ws = dw.workspace_for(w)
    first = dw.run(w, d, ws=ws).to_numpy()
    for _ in range(3):
        again = dw.run(w, d, ws=ws).to_numpy()
        for k in first:
            assert np.array_equal(first[k], again[k]), k
    n = sv.workspace_bytes(w.rows, w.batch, w.vocab, w.max_len)
    assert int(ws[: n].sum().item()) != 0  # scratch is in use, counters were reset by the kernels


@pytest.mark.parametrize("idx", [4, 5])
def test_graph_replay_equals_eager(idx):
    """The benchmark replays the step from a CUDA graph: replayed outputs equal the eager call's bit for bit."""
    w = wl.config(idx)
    d = dw.DeviceInputs.from_workload(w)
    eager = dw.run(w, d, out=dw.outputs_for(w), ws=dw.workspace_for(w))
    torch.cuda.synchronize()
    want = eager.to_numpy()
    out, ws = dw.outputs_for(w), dw.workspace_for(w)
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        dw.run(w, d, out=out, ws=ws)  # per-device caches filled outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        dw.run(w, d, out=out, ws=ws)
    torch.cuda.synchronize()
    for k in out.__dict__:
        t = getattr(out, k)
        if t is not None:
            t.fill_(-7)  # the replays must rewrite every output
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    got = out.to_numpy()
    n = int(want["commit_cu"][-1])  # the KV-commit lists are written up to the committed count only
    for k in want:
        if k in ("commit_src_slot", "commit_dst_pos"):
            assert np.array_equal(want[k][:n], got[k][:n]), k
        else:
            assert np.array_equal(want[k], got[k]), k
