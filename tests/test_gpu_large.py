"""Inputs past 2^31 and 2^32 bytes: every address the kernels form is 64-bit.

A 1024-request rejection chain of 16 rows over V = 151936 bf16 logits (16384
rows, 4.98 GB; q 9.96 GB of fp32) is generated on the device with a seed and
verified end to end.  The requests whose rows straddle the 2^31- and 2^32-byte
marks of the logits, the first and the last request and a few at random are
then compared with the oracle on their own rows (as a ragged batch of just
those requests), under the parity rule; the row statistics of rows around the
marks are compared with the oracle too.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import oracle  # noqa: E402
from reject_row_vocab_gb300 import _build  # noqa: E402

_build.build()
from reject_row_vocab_gb300 import specverify as sv  # noqa: E402
from tests.gpu_compare import compare, oracle_outputs  # noqa: E402
from tests.helpers import chain_workload  # noqa: E402

B, M, V = 1024, 15, 151936
L = M + 1
R = B * L
CHUNK = 1024  # rows generated at a time


def _need_memory(gb: float):
    free, _ = torch.cuda.mem_get_info()
    if free < gb * 2**30:
        pytest.skip("needs %.0f GB of free device memory" % gb)


@pytest.fixture(scope="module")
def big_chain():
    _need_memory(40)
    g = torch.Generator(device="cuda")
    g.manual_seed(2024)
    logits = torch.empty((R, V), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((R, V), dtype=torch.float32, device="cuda")
    ids = torch.zeros(R, dtype=torch.int32, device="cuda")
    for r0 in range(0, R, CHUNK):
        x = torch.randn((CHUNK, V), generator=g, device="cuda") * 3.0
        logits[r0:r0 + CHUNK] = x.to(torch.bfloat16)
        noisy = logits[r0:r0 + CHUNK].float() + 1.5 * torch.randn((CHUNK, V), generator=g, device="cuda")
        q[r0:r0 + CHUNK] = torch.softmax(noisy, dim=1)
        drafts = torch.multinomial(q[r0:r0 + CHUNK], 1, generator=g).view(-1).to(torch.int32)
        # row j of a request tests the draft drawn from its own q; the anchor slot of each request stays 0
        rows = torch.arange(r0, r0 + CHUNK, device="cuda")
        nxt = rows + 1
        keep = (rows % L) != L - 1
        ids[nxt[keep]] = drafts[keep]
        del x, noisy
    T = torch.rand(B, generator=g, device="cuda") * 0.7 + 0.5
    ua = torch.rand(R, generator=g, device="cuda")
    uf = torch.rand(B, generator=g, device="cuda")
    row_slots = torch.randperm(1 << 20, generator=g, device="cuda")[:R].to(torch.int64)
    seq_lens = torch.randint(128, 4097, (B,), generator=g, device="cuda").to(torch.int64)
    out = sv.rejection_chain(logits, ids, M, q, T, ua, uf, row_slots=row_slots, seq_lens=seq_lens)
    torch.cuda.synchronize()
    yield dict(logits=logits, q=q, ids=ids, T=T, ua=ua, uf=uf, row_slots=row_slots, seq_lens=seq_lens,
               out=out.to_numpy())
    del logits, q
    torch.cuda.empty_cache()


def _requests():
    mark31 = (1 << 31) // (V * 2)  # rows whose logits cross the 2^31- and 2^32-byte marks
    mark32 = (1 << 32) // (V * 2)
    picks = {0, B - 1, mark31 // L, (mark31 + 1) // L, mark32 // L, (mark32 + 1) // L}
    rng = np.random.default_rng(7)
    picks.update(int(b) for b in rng.integers(0, B, 4))
    return sorted(picks)


def test_rows_past_the_32_bit_marks_match_the_oracle(big_chain):
    d = big_chain
    picks = _requests()
    rows = np.concatenate([np.arange(b * L, (b + 1) * L) for b in picks])
    lg = d["logits"][torch.from_numpy(rows).cuda()].contiguous()
    bits = lg.view(torch.int16).cpu().numpy().view(np.uint16)
    qh = d["q"][torch.from_numpy(rows).cuda()].cpu().numpy()
    cu = np.arange(0, (len(picks) + 1) * L, L, dtype=np.int32)
    slots = d["row_slots"].cpu().numpy()[rows]
    w = chain_workload(bits, "bf16", cu, d["ids"].cpu().numpy()[rows], q=qh,
                       T=d["T"].cpu().numpy()[picks], ua=d["ua"].cpu().numpy()[rows], uf=d["uf"].cpu().numpy()[picks],
                       max_len=L, kind="rejection_ragged", row_slots=slots,
                       seq_lens=d["seq_lens"].cpu().numpy()[picks], name="beyond_4GB_rejection_chain")
    o = d["out"]
    cu_big = o["commit_cu"].astype(np.int64)
    g = {k: [] for k in ("accept_len", "num_out", "bonus", "out_tokens", "accept_rows", "status",
                         "commit_src_slot", "commit_dst_pos")}
    for k, b in enumerate(picks):
        for key in ("accept_len", "num_out", "bonus", "status"):
            g[key].append(o[key][b])
        g["out_tokens"].append(o["out_tokens"][b])
        ar = o["accept_rows"][b].astype(np.int64)
        g["accept_rows"].append(np.where(ar >= 0, ar - b * L + k * L, -1).astype(np.int32))
        n = int(o["num_out"][b])
        g["commit_src_slot"].append(o["commit_src_slot"][cu_big[b]:cu_big[b] + n])
        g["commit_dst_pos"].append(o["commit_dst_pos"][cu_big[b]:cu_big[b] + n])
    g = {k: (np.concatenate(v) if k.startswith("commit_") else np.asarray(v)) for k, v in g.items()}
    g["commit_cu"] = np.concatenate([[0], np.cumsum(g["num_out"].astype(np.int64))]).astype(np.int32)
    compare(w, g, oracle_outputs(w))
    # the whole batch commits consistently
    assert cu_big[0] == 0 and np.array_equal(np.diff(cu_big), o["num_out"])


def test_row_statistics_past_the_32_bit_marks(big_chain):
    d = big_chain
    mark31 = (1 << 31) // (V * 2)
    mark32 = (1 << 32) // (V * 2)
    rows = np.array(sorted({0, mark31 - 1, mark31, mark31 + 1, mark32 - 1, mark32, mark32 + 1, R - 1}))
    T = torch.full((R,), 0.8, dtype=torch.float32, device="cuda")
    r = sv.row_stats(d["logits"], row_temp=T)
    torch.cuda.synchronize()
    bits = d["logits"][torch.from_numpy(rows).cuda()].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.row_stats(bits, "bf16", row_temp=np.full(len(rows), 0.8, np.float32))
    assert np.array_equal(r["argmax"].cpu().numpy()[rows], ref["argmax"])
    assert np.array_equal(r["max"].cpu().numpy()[rows].astype(np.float64), ref["max"])
    z = r["z"].cpu().numpy()[rows]
    assert np.all(np.abs(z - ref["z"]) <= 2e-6 * ref["z"])
