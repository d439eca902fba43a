import os
import sys

ROOT = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(ROOT)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libspecverify")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Parity counts of every CUDA-vs-oracle comparison of the run (printed without -s)."""
    mod = sys.modules.get("tests.gpu_compare")
    rep = getattr(mod, "REPORT", None) if mod else None
    if not rep:
        return
    tot = {k: sum(r[k] for _, r in rep) for k in ("requests", "exact", "draw_flagged", "test_flagged", "differ",
                                                  "mismatch")}
    terminalreporter.write_line(
        "parity: %d comparisons, %d requests: %d exact, %d with only the final draw within 1e-6 of a CDF edge, "
        "%d with an acceptance test within 1e-6 (compared up to it); %d flagged differ from the oracle; "
        "%d mismatches" % (len(rep), tot["requests"], tot["exact"], tot["draw_flagged"], tot["test_flagged"],
                           tot["differ"], tot["mismatch"]))
    full = [(n, r) for n, r in rep if n.startswith("c") and "_" in n and n[1].isdigit()]
    for n, r in full:
        terminalreporter.write_line("parity %s: %d requests, %d exact, %d draw-flagged, %d test-flagged, %d differ"
                                    % (n, r["requests"], r["exact"], r["draw_flagged"], r["test_flagged"],
                                       r["differ"]))
