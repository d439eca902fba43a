"""Sample-then-match verification on the GPU vs the oracle.

Same bar as the chains: decisions, lengths, tokens, commit lists and status
bits bit-exact on every request not within 1e-6 of a sampling boundary.
"""
import dataclasses

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from reject_row_vocab_gb300 import _build  # noqa: E402

_build.build()
from reject_row_vocab_gb300 import device_workload as dw  # noqa: E402
from reject_row_vocab_gb300 import workload as wl  # noqa: E402
from tests.gpu_compare import compare, oracle_outputs  # noqa: E402


def as_match(w):
    return dataclasses.replace(w, kind="sample_match_chain", q=None, name=w.name + "_match")


def check(w):
    d = dw.DeviceInputs.from_workload(w)
    g = dw.run(w, d, ws=dw.workspace_for(w)).to_numpy()
    torch.cuda.synchronize()
    o = oracle_outputs(w)
    r = compare(w, g, o)
    print(w.name, r, "mean accept", float(np.mean(o["accept_len"])))
    return g, o


@pytest.mark.parametrize("batch,m,vocab,dtype,T,boost,sigma", [
    (6, 4, 300, "f32", 0.9, 4.0, 1.0),
    (8, 7, 2053, "bf16", 0.8, 6.0, 2.0),       # ragged vocab (tail vector)
    (5, 6, 20011, "bf16", 1.0, 8.0, 1.5),
    (4, 3, 4099, "f32", 0.5, 10.0, 1.0),
    (16, 15, 65536, "bf16", 1.0, 9.0, 2.0),
])
def test_match_chain_matches_oracle(batch, m, vocab, dtype, T, boost, sigma):
    w = wl.rejection_chain(batch=batch, m=m, vocab=vocab, dtype=dtype, boost=boost, sigma=sigma, temperature=T,
                           noise_sigma=0.2, seed=batch * 31 + vocab)
    check(as_match(w))


def test_match_greedy_mixed_and_degenerate():
    w = as_match(wl.rejection_chain(batch=8, m=4, vocab=1000, dtype="f32", boost=5.0, sigma=1.0, noise_sigma=0.2,
                                    seed=41))
    T, ids, x = w.temperature.copy(), w.verify_ids.copy(), w.logits.copy()
    L = w.max_len
    T[1] = 0.0                       # greedy request
    ids[2 * L + 1] = 5000            # request 2 tests an out-of-range id at row 0
    x[3 * L + 0, :] = -np.inf        # request 3: no usable logit at row 0
    x[4 * L + 1, 7] = np.nan         # request 4: a NaN entry
    check(dataclasses.replace(w, temperature=T, verify_ids=ids, logits=x))


def test_full_size_dflash_block_shape():
    w = as_match(wl.config(4))
    g, o = check(w)
