"""Tree-verify inputs built on the GPU vs the oracle (exact integers)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from oracle import tree_build as tb  # noqa: E402
from reject_row_vocab_gb300 import _build  # noqa: E402

_build.build()
from reject_row_vocab_gb300 import specverify as sv  # noqa: E402
from reject_row_vocab_gb300 import workload as wl  # noqa: E402


def _check(par, sl):
    B, N = par.shape
    g = sv.build_tree(torch.from_numpy(par).cuda(), torch.from_numpy(sl).cuda())
    g = {k: v.cpu().numpy() for k, v in g.items()}
    for b in range(B):
        o = tb.build(par[b].tolist(), int(sl[b]), b)
        assert g["positions"][b].tolist() == o["positions"], b
        assert np.array_equal(g["mask"][b], np.array(o["mask"], np.uint8)), b
        assert g["retrieve_index"][b].tolist() == o["retrieve_index"]
        assert g["first_child"][b].tolist() == o["first_child"], b
        assert g["next_sibling"][b].tolist() == o["next_sibling"], b
        assert int(g["status"][b]) == o["status"], b


@pytest.mark.parametrize("B,N", [(1, 1), (3, 6), (16, 17), (8, 64), (4, 300), (2, 1024)])
def test_random_trees(B, N):
    rng = np.random.default_rng(B * 7 + N)
    par = np.empty((B, N), np.int32)
    for b in range(B):
        par[b, 0] = -1
        for i in range(1, N):
            # deep chains, wide fans and mixtures
            par[b, i] = i - 1 if b % 3 == 0 else (0 if b % 3 == 1 else int(rng.integers(max(0, i - 4), i)))
    sl = rng.integers(0, 5000, size=B).astype(np.int64)
    _check(par, sl)


def test_eagle2_tree_workload_and_invalid_trees():
    w = wl.config(3, mode="greedy_tree")
    par = np.ascontiguousarray(w.parents, dtype=np.int32)
    _check(par, np.asarray(w.seq_lens, dtype=np.int64))
    bad = par.copy()
    bad[1, 0] = 0        # root with a parent
    bad[2, 5] = 7        # a parent after its child
    bad[3, 3] = -1       # a second root
    _check(bad, np.zeros(len(bad), np.int64))
