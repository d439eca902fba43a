"""DSpark verify-length allocation on the GPU against the oracle (exact integers)."""
import json
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from oracle import dspark  # noqa: E402
from reject_row_vocab_gb300 import _build  # noqa: E402

_build.build()
from reject_row_vocab_gb300 import specverify as sv  # noqa: E402

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "dspark_scheduler_example.json")))


def _gpu(survival, k, min_len=1, max_len=None, eps=0.0, pad=0):
    s = np.asarray(survival, dtype=np.float32)
    R, D = s.shape
    buf = np.zeros((R, D + pad), np.float32)
    buf[:, :D] = s
    t = torch.from_numpy(buf).cuda()[:, :D]
    out = sv.dspark_verify_lens(t, k, min_len=min_len, max_len=max_len if max_len else D + 1, eps=eps)
    return out.cpu().numpy().tolist()


def test_page_example():
    g = GOLD["allocation"]
    assert _gpu(g["survival"], g["budget"]) == g["verify_lens"]


@pytest.mark.parametrize("R,D", [(1, 1), (2, 3), (7, 5), (64, 8), (256, 16), (300, 7), (1024, 32)])
def test_random_with_ties_matches_oracle(R, D):
    rng = np.random.default_rng(R * 100 + D)
    for trial in range(3):
        conf = rng.choice([0.5, 0.7, 0.9, 0.95, 1.0], size=(R, D)).astype(np.float32)
        surv = np.cumprod(conf, axis=1, dtype=np.float32)
        if trial == 2:
            surv[rng.random((R, D)) < 0.05] = np.nan
        k = int(rng.integers(0, R * D + 3))
        eps = [0.0, 0.3, 0.0][trial]
        max_len = int(rng.integers(1, D + 2))
        want = dspark.verify_lens(surv.astype(np.float64).tolist(), k, 1, max_len, eps)
        assert _gpu(surv, k, 1, max_len, eps, pad=trial) == want


def test_workspace_is_left_clean_for_reuse():
    rng = np.random.default_rng(3)
    surv = np.cumprod(rng.uniform(0.5, 1.0, size=(40, 6)).astype(np.float32), axis=1)
    ws = sv.dspark_workspace(40, "cuda")
    a = sv.dspark_verify_lens(torch.from_numpy(surv).cuda(), 50, ws=ws).cpu().numpy().tolist()
    b = sv.dspark_verify_lens(torch.from_numpy(surv).cuda(), 50, ws=ws).cpu().numpy().tolist()
    assert a == b == dspark.verify_lens(surv.astype(np.float64).tolist(), 50)
    assert int(ws.sum().item()) == 0


def test_degenerate_shapes():
    # no drafts: every request verifies just its anchor (clamped into [min_len, max_len])
    t = torch.zeros((5, 0), dtype=torch.float32, device="cuda")
    assert sv.dspark_verify_lens(t, 3, min_len=1, max_len=4).cpu().tolist() == [1] * 5
    assert sv.dspark_verify_lens(torch.ones((3, 2), device="cuda"), 0, min_len=2, max_len=3).cpu().tolist() == [2] * 3
