"""Host-side pieces of bench.py: L2-flush choice, config text, traffic record gating (no GPU)."""
import json
import os
import sys
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _w(name, kind, logit_bytes):
    return types.SimpleNamespace(name=name, kind=kind, batch=1, rows=1, vocab=1, max_len=1, dtype="bf16",
                                 meta={"seed": 1}, logit_bytes=lambda: logit_bytes)


def test_flush_choice_follows_l2_size():
    import bench
    small, large = _w("c3_greedy_tree", "greedy_tree", 69_771_264), _w("c4_dflash_block", "rejection_chain",
                                                                         311_164_928)
    auto = bench.parse_args([])
    assert bench.flush_wanted(auto, small) and not bench.flush_wanted(auto, large)
    assert bench.flush_wanted(bench.parse_args(["--flush-l2", "on"]), large)
    assert not bench.flush_wanted(bench.parse_args(["--flush-l2", "off"]), small)
    assert bench.FLUSH_BYTES > 1.9 * bench.L2_BYTES
    assert "flushed" in bench.describe(small, True)["l2"]
    assert "larger than L2" in bench.describe(large, False)["l2"]
    assert "not flushed" in bench.describe(small, False)["l2"]


def test_traffic_record_applies_only_to_its_workload_and_source(tmp_path, monkeypatch):
    """The ncu traffic figure is used only for its own workload and only while the kernel source it was
    captured from is unchanged (checked on a copy of the tree)."""
    import hashlib
    import shutil

    import bench
    for rel in bench.STATS_SOURCES:
        os.makedirs(os.path.dirname(tmp_path / rel), exist_ok=True)
        shutil.copy(os.path.join(ROOT, rel), tmp_path / rel)
    h = hashlib.sha256()
    for rel in bench.STATS_SOURCES:
        h.update(open(tmp_path / rel, "rb").read())
    os.makedirs(tmp_path / "profiles")
    rec = {"workload_name": "c4_dflash_block", "bytes_per_full_launch": 123.0, "source_sha256": h.hexdigest()}
    with open(tmp_path / "profiles" / "traffic.json", "w") as f:
        json.dump(rec, f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = rec["workload_name"]
    assert bench.stats_traffic(_w(base, "rejection_chain", 1)) == 123.0
    assert bench.stats_traffic(_w(base + "_sparse_q16", "rejection_chain_sparse", 1)) == 123.0
    assert bench.stats_traffic(_w(base + "_sample_match", "sample_match_chain", 1)) is None
    assert bench.stats_traffic(_w("c3_greedy_tree", "greedy_tree", 1)) is None
    with open(tmp_path / bench.STATS_SOURCES[0], "a") as f:
        f.write("// changed\n")
    assert bench.stats_traffic(_w(base, "rejection_chain", 1)) is None  # the kernel changed since the capture


def test_aux_modes_inputs_and_reference_arm(capsys):
    import bench
    x = bench.aux_inputs("dspark")
    assert x["survival"].shape == (256, 15) and x["survival"].dtype.name == "float32"
    assert (x["survival"][:, 1:] <= x["survival"][:, :-1]).all()  # running products only fall
    t = bench.aux_inputs("tree-build")
    par = t["parents"]
    assert par.shape == (64, 64) and (par[:, 0] == -1).all()
    assert all((par[:, i] >= 0).all() and (par[:, i] < i).all() for i in range(1, 64))
    assert bench.aux_config("dspark", x)["workload"] == "dspark_schedule_r256_d15"
    for kind in ("dspark", "tree-build"):
        bench.main(["--impl", "reference", "--kernel", kind, "--steps", "2", "--warmup", "1"])
        line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
        assert line["impl"] == "reference" and line["steps"] == 2 and line["value"] > 0
        assert line["metric"] == bench.AUX[kind]["metric"] and line["warmup"] == 3


def test_step_reference_arm_line(capsys):
    """The reference arm of the verify step (the oracle on the host cores) prints one line with the contract's keys:
    its own value in cpu_baseline and e2e, no host-device bytes, the workload named in config."""
    import bench
    bench.main(["--impl", "reference", "--config", "1", "--steps", "2", "--warmup", "1"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 2 and line["value"] > 0
    assert line["warmup"] == 3  # the bench runs at least three warm-up steps and reports what it ran
    assert line["config"]["workload"] == "c1_greedy_chain" and line["higher_is_better"] is True
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    e = line["e2e"]
    assert e["value"] == line["value"] and e["unit"] == line["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_stats_event_slots():
    import bench
    assert bench.stats_event_slots(5, 1) == [0, 1, 2, 3, 4]
    assert bench.stats_event_slots(25, 10) == [0] + [None] * 9 + [1] + [None] * 9 + [2] + [None] * 4
    assert bench.stats_event_slots(3, 10) == [0, None, None]
    slots = bench.stats_event_slots(100, 7)
    used = [x for x in slots if x is not None]
    assert used == list(range(len(used))) and len(used) == 15
