"""The C-ABI library loads and exports every symbol its header declares; host-side
argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="module")
def lib():
    from reject_row_vocab_gb300 import _build, specverify
    _build.build()
    return specverify.load_library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\*?\s+\*?(spec_verify_[a-z_]+)\s*\(",
                                 text, re.M)))


def test_header_declares_the_five_entry_points():
    names = declared_functions()
    for n in ("spec_verify_greedy_chain", "spec_verify_greedy_tree", "spec_verify_rejection_chain",
              "spec_verify_rejection_ragged", "spec_verify_target_only_tree"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from reject_row_vocab_gb300 import specverify
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    assert set(specverify.ENTRY_POINTS) <= set(names)


def test_status_strings_and_workspace_size(lib):
    for code in range(8):
        assert lib.spec_verify_status_string(code)
    small = lib.spec_verify_workspace_bytes(5, 1, 32000, 5)
    big = lib.spec_verify_workspace_bytes(1024, 64, 151936, 16)
    assert 0 < small < big
    assert big % 256 == 0
    # a sparse q's candidate lists are read in place: its workspace is the dense one, whatever num_cands is
    lib.spec_verify_sparse_workspace_bytes.restype = ctypes.c_size_t
    lib.spec_verify_sparse_workspace_bytes.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                                       ctypes.c_int32, ctypes.c_int32]
    for k in (1, 16, 1024):
        assert lib.spec_verify_sparse_workspace_bytes(1024, 64, 151936, 16, k) == big


def _out_struct(addr=0x10000):
    from reject_row_vocab_gb300.specverify import SvOut
    return SvOut(*([addr] * 9))


def test_host_validation_without_gpu(lib):
    """Argument errors return before anything is enqueued, so they need no device."""
    P = ctypes.c_void_p
    fake = P(0x100000)  # aligned, never dereferenced on the host
    out = _out_struct()
    null = None
    ws = P(0x200000)
    # NULL logits
    assert lib.spec_verify_greedy_chain(null, 1, 64, 2, 3, 64, fake, null, null, ctypes.byref(out), ws, 1 << 30,
                                        null) == 1
    # bad dtype
    assert lib.spec_verify_greedy_chain(fake, 7, 64, 2, 3, 64, fake, null, null, ctypes.byref(out), ws, 1 << 30,
                                        null) == 3
    # ld < vocab
    assert lib.spec_verify_greedy_chain(fake, 1, 32, 2, 3, 64, fake, null, null, ctypes.byref(out), ws, 1 << 30,
                                        null) == 2
    # misaligned base pointer and row stride
    assert lib.spec_verify_greedy_chain(P(0x100002), 1, 64, 2, 3, 64, fake, null, null, ctypes.byref(out), ws,
                                        1 << 30, null) == 4
    assert lib.spec_verify_greedy_chain(fake, 1, 67, 2, 3, 64, fake, null, null, ctypes.byref(out), ws, 1 << 30,
                                        null) == 4
    # commit_src_slot requested without row_slots
    assert lib.spec_verify_greedy_chain(fake, 1, 64, 2, 3, 64, fake, null, null, ctypes.byref(out), ws, 1 << 30,
                                        null) == 1
    out2 = _out_struct()
    out2.commit_src_slot = None
    out2.commit_dst_pos = None
    # workspace too small / misaligned
    assert lib.spec_verify_greedy_chain(fake, 1, 64, 2, 3, 64, fake, null, null, ctypes.byref(out2), ws, 16,
                                        null) == 6
    assert lib.spec_verify_greedy_chain(fake, 1, 64, 2, 3, 64, fake, null, null, ctypes.byref(out2), P(0x200010),
                                        1 << 30, null) == 6
    # trees: too many nodes, a half-given sibling list, bad threshold
    assert lib.spec_verify_greedy_tree(fake, 1, 64, 2, 4096, 64, fake, fake, null, null, null, null,
                                       ctypes.byref(out2), ws, 1 << 30, null) == 2
    assert lib.spec_verify_greedy_tree(fake, 1, 64, 2, 8, 64, fake, fake, fake, null, null, null,
                                       ctypes.byref(out2), ws, 1 << 30, null) == 1
    assert lib.spec_verify_target_only_tree(fake, 1, 64, 2, 8, 64, fake, fake, null, null, fake,
                                            ctypes.c_float(1.0), ctypes.c_float(0.0), fake, fake, null, null,
                                            ctypes.byref(out2), ws, 1 << 30, null) == 2
    for th_single, th_acc in ((1.0, float("inf")), (float("nan"), 1.0), (1.0, -0.5)):
        assert lib.spec_verify_target_only_tree(fake, 1, 64, 2, 8, 64, fake, fake, null, null, fake,
                                                ctypes.c_float(th_single), ctypes.c_float(th_acc), fake, fake, null,
                                                null, ctypes.byref(out2), ws, 1 << 30, null) == 2
    # rejection: q missing, q stride misaligned
    assert lib.spec_verify_rejection_chain(fake, 1, 64, 2, 3, 64, fake, null, 64, fake, fake, fake, null, null,
                                           ctypes.byref(out2), ws, 1 << 30, null) == 1
    assert lib.spec_verify_rejection_chain(fake, 1, 64, 2, 3, 64, fake, fake, 65, fake, fake, fake, null, null,
                                           ctypes.byref(out2), ws, 1 << 30, null) == 4
    # ragged: max_len < 1
    assert lib.spec_verify_rejection_ragged(fake, 1, 64, 2, 8, 0, 64, fake, fake, fake, 64, fake, fake, fake, null,
                                            null, ctypes.byref(out2), ws, 1 << 30, null) == 2


def test_no_alloc_entry_checks_arguments_before_any_cuda_call(lib):
    """Refusals of the no-allocation entry come before its scratch lookup and its counter clear: without a GPU
    they still return the argument's own status, not SV_ERR_CUDA."""
    P = ctypes.c_void_p
    fake, null = P(0x100000), None
    out = _out_struct()
    out.commit_src_slot = None
    out.commit_dst_pos = None
    fn = lib.spec_verify_rejection_chain_noalloc
    I32, I64 = ctypes.c_int32, ctypes.c_int64
    fn.argtypes = [P, ctypes.c_int, I64, I32, I32, I32, P, P, I64, P, P, P, P, P, P, P]
    fn.restype = ctypes.c_int

    def call(verify_ids=fake, q=fake, ldq=64, dtype=1, batch=2, vocab=64):
        return fn(fake, dtype, 64, batch, 3, vocab, verify_ids, q, ldq, fake, fake, fake, null, null,
                  ctypes.byref(out), null)

    assert call(verify_ids=null) == 1
    assert call(q=null) == 1
    assert call(ldq=65) == 4
    assert call(dtype=4) == 3
    assert call(batch=4096, vocab=1 << 20) == 6


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from reject_row_vocab_gb300 import specverify
    monkeypatch.setattr(specverify, "_lib", None)
    monkeypatch.setattr(specverify, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        specverify.load_library()


def test_host_validation_of_the_later_entry_points(lib):
    """Sparse q, sample-then-match and the tree build refuse bad arguments before touching a GPU."""
    P = ctypes.c_void_p
    fake, ws, null = P(0x100000), P(0x200000), None
    out = _out_struct()
    out.commit_src_slot = None
    out.commit_dst_pos = None
    o = ctypes.byref(out)

    def sparse(batch=2, m=3, cand_ids=fake, cand_probs=fake, k=4, ldc=4, dtype=1):
        return lib.spec_verify_rejection_chain_sparse(fake, dtype, 64, batch, m, 64, fake, cand_ids, cand_probs, k,
                                                      ldc, fake, fake, fake, null, null, o, ws, 1 << 30, null)

    assert sparse(cand_ids=null) == 1
    assert sparse(cand_probs=null) == 1
    assert sparse(k=0) == 2
    assert sparse(k=1025, ldc=2048) == 2      # more candidates per row than the sampler holds
    assert sparse(k=8, ldc=4) == 2            # row stride shorter than the list
    assert sparse(batch=65536) == 2
    assert sparse(m=-1) == 2
    assert sparse(dtype=5) == 3

    def match(batch=2, m=3, u=fake, dtype=1, ld=64):
        return lib.spec_verify_sample_match_chain(fake, dtype, ld, batch, m, 64, fake, fake, u, null, null, o, ws,
                                                  1 << 30, null)

    assert match(u=null) == 1
    assert match(batch=65536) == 2
    assert match(m=-1) == 2
    assert match(dtype=9) == 3
    assert match(ld=68) == 4                  # bf16 rows of 136 bytes: not a multiple of 16

    def tree(batch=2, nodes=8, parents=fake):
        return lib.spec_verify_build_tree(parents, null, batch, nodes, fake, fake, fake, fake, fake, fake, null)

    assert tree(parents=null) == 1
    assert tree(nodes=0) == 2
    assert tree(nodes=1025) == 2              # above the per-request node bound
    assert tree(batch=-1) == 2
    assert tree(batch=0) == 0                 # nothing to do, nothing enqueued
