"""The oracle's pins fail on planted mistakes.

Each case copies the oracle, plants one plausible mistake in the copy (a
swapped acceptance test, a dropped temperature, an unclamped residual, a wrong
tie-break, a misread threshold rule, a wrong scheduling order, ...), builds it
with the host compiler into a temporary directory and runs the pin tests
against it in a child process: at least one pin must fail there.  The oracle
itself is never modified.
"""
import os
import shutil
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")
PINS = ["tests/test_oracle_pins.py", "tests/test_oracle_gaps.py"]

# name -> [(text in the oracle, planted replacement), ...]; each text occurs exactly once
MUTATIONS = {
    "acceptance test swapped, u*p < q": [("return u * q < p;", "return u * p < q;")],
    "argmax ties go to the highest index": [("if (l > r.M) {", "if (l >= r.M) {")],
    "temperature dropped from the softmax": [
        ("Z += std::exp((l - r.M) / T);", "Z += std::exp(l - r.M);"),
        ("return std::exp((l - r.M) / r.T) / r.Z;", "return std::exp(l - r.M) / r.Z;"),
    ],
    "residual taken as q - p": [
        ("w[v] = std::max(0.0, p[v] - static_cast<double>(q[v]));",
         "w[v] = std::max(0.0, static_cast<double>(q[v]) - p[v]);"),
    ],
    "residual not clamped at 0": [
        ("w[v] = std::max(0.0, p[v] - static_cast<double>(q[v]));", "w[v] = p[v] - static_cast<double>(q[v]);"),
    ],
    "inverse CDF target not scaled by the total": [("double t = u * S;", "double t = u;")],
    "greedy tree accepts a child that is not the argmax": [("if (tok[k] == st.argmax) {", "if (tok[k] != st.argmax) {")],
    "theta_acc multiplies the cumulative mass": [
        ("if (u < c / a.th_acc || pk >= a.th_single) {", "if (u < c * a.th_acc || pk >= a.th_single) {"),
    ],
    "theta_single compared strictly": [
        ("if (u < c / a.th_acc || pk >= a.th_single) {", "if (u < c / a.th_acc || pk > a.th_single) {"),
    ],
    "target-only stop draw keeps the children": [("for (int32_t t : seen) w[t] = 0.0;", "for (int32_t t : seen) (void)t;")],
    "cumulative mass taken before the child": [
        ("if (u < c / a.th_acc || pk >= a.th_single) {", "if (u < (c - pk) / a.th_acc || pk >= a.th_single) {"),
    ],
    "final token drawn from the row before the stop": [
        ("const int64_t s = start + j;", "const int64_t s = start + (j > 0 ? j - 1 : 0);"),
    ],
    "acceptance gap measured as |u - q/p|": [
        ("std::fabs(u - p / qd)", "std::fabs(u - qd / p)"),
    ],
    "committed rows of a request written in reverse": [
        ("int64_t dst = o.commit_cu[b] + k;", "int64_t dst = o.commit_cu[b + 1] - 1 - k;"),
    ],
    "row statistics report p at the argmax instead of the probe": [
        ("pv = prob(st, lg.at(r, probe[r]));", "pv = prob(st, lg.at(r, st.argmax));"),
    ],
    "row statistics flag nothing for NaN or +inf": [
        ("out_flags[r] = st.nonfinite ? kNonFinite : 0u;", "out_flags[r] = 0u;"),
    ],
    "children found from the node after the current one only": [
        ("for (int32_t i = cur + 1; i < a.N; ++i)\n      if (par[i] == cur) kids.push_back(i);",
         "for (int32_t i = cur + 2; i < a.N; ++i)\n      if (par[i] == cur) kids.push_back(i);"),
    ],
    "tree validation accepts a parent that is not before its node": [
        ("if (par[i] < 0 || par[i] >= i) return false;", "if (par[i] < 0 || par[i] >= a.N) return false;"),
    ],
    "chain residual fallback to p not flagged": [
        ("  if (v < 0) {\n    rr.status |= kResidualEmpty;\n", "  if (v < 0) {\n"),
    ],
    "repeated sibling token not flagged": [("          rr.status |= kDupSibling;\n", "")],
    "invalid tree not flagged": [("  if (!ok_tree) rr.status |= kBadTree;", "  (void)ok_tree;")],
    "invalid row range not flagged": [("    rr.status |= kBadLayout;", "")],
    "destination position one past the committed offset": [
        ("o.commit_dst_pos[dst] = seq_lens[b] + k;", "o.commit_dst_pos[dst] = seq_lens[b] + k + 1;"),
    ],
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_fail_on_a_planted_mistake(name, tmp_path):
    src = open(SRC).read()
    for old, new in MUTATIONS[name]:
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new)
    cpp = tmp_path / "oracle_planted.cpp"
    cpp.write_text(src)
    lib = str(tmp_path / "liboracle_planted.so")
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", str(cpp), "-o", lib])
    code = textwrap.dedent("""
        import sys
        sys.path.insert(0, %r)
        import oracle
        oracle._LIB = %r
        oracle.build = lambda force=False: %r
        import pytest
        sys.exit(pytest.main(["-q", "-x", "-p", "no:cacheprovider", *%r]))
    """) % (ROOT, lib, lib, PINS)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    # exit status 1: tests ran and one failed (0 would mean every pin passed; anything else a crash or an error)
    assert r.returncode == 1, (name, r.returncode, r.stdout[-3000:], r.stderr[-2000:])


# The Python oracles: name -> (file under oracle/, [(text, planted replacement)], pin files)
PY_MUTATIONS = {
    "DSpark budget sorts the survival scores ascending": (
        "dspark.py",
        [("reverse=True)\n    best_k, best = 0, -math.inf", "reverse=False)\n    best_k, best = 0, -math.inf")],
        ["tests/test_dspark_oracle.py"]),
    "DSpark budget ties keep the larger K": (
        "dspark.py", [("        if score > best:", "        if score >= best:")], ["tests/test_dspark_oracle.py"]),
    "DSpark top-K orders ties by request before position": (
        "dspark.py", [("cands.append((-key, j, r, s))", "cands.append((-key, r, j, s))")],
        ["tests/test_dspark_oracle.py"]),
    "sample-then-match accepts a mismatching draft": (
        "match.py", [("            if d != t:", "            if d == t:")], ["tests/test_match_oracle.py"]),
    "tree depth from the previous index instead of the parent": (
        "tree_build.py", [("depth[i] = depth[parents[i]] + 1", "depth[i] = depth[i - 1] + 1")],
        ["tests/test_tree_build_oracle.py"]),
    "next sibling is the last one instead of the next": (
        "tree_build.py", [("later[0] if later else -1", "later[-1] if later else -1")],
        ["tests/test_tree_build_oracle.py"]),
    "sparse q keeps the last of repeated ids instead of their sum": (
        "__init__.py", [("np.add.at(q, (rr[ok], ids[ok]), pr[ok])", "q[rr[ok], ids[ok]] = pr[ok]")],
        ["tests/test_sparse_oracle.py"]),
    "DSpark verify lengths leave out the anchor row": (
        "dspark.py", [("return [min(max(1 + e, min_len), max_len) for e in extra]",
                       "return [min(max(e, min_len), max_len) for e in extra]")],
        ["tests/test_dspark_oracle.py"]),
    "sparse q flags padding ids as out of range": (
        "__init__.py", [("bad = np.any((ids != -1) & ~ok, axis=1)", "bad = np.any(~ok, axis=1)")],
        ["tests/test_sparse_oracle.py"]),
    "parity rule lets a close final draw exempt the whole request": (
        "parity.py", [("            for k in (\"accept_len\", \"num_out\", \"accept_rows\", \"status\"):",
                       "            for k in ():")],
        ["tests/test_parity_rule.py"]),
    "parity rule exempts every acceptance test": (
        "parity.py", [("close = np.nonzero(test_gap[b] < tol)[0]", "close = np.nonzero(test_gap[b] < 1.0)[0]")],
        ["tests/test_parity_rule.py"]),
}


@pytest.mark.parametrize("name", sorted(PY_MUTATIONS))
def test_python_oracle_pins_fail_on_a_planted_mistake(name, tmp_path):
    fname, edits, pins = PY_MUTATIONS[name]
    pkg = tmp_path / "oracle"
    shutil.copytree(os.path.join(ROOT, "oracle"), pkg,
                    ignore=shutil.ignore_patterns("*.so", "*.tmp*", "__pycache__"))
    path = pkg / fname
    src = path.read_text()
    for old, new in edits:
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new)
    path.write_text(src)
    code = textwrap.dedent("""
        import sys
        sys.path.insert(0, %r)
        sys.path.insert(0, %r)
        import oracle, oracle.dspark, oracle.match, oracle.tree_build, oracle.parity
        assert oracle.__file__.startswith(%r), oracle.__file__
        import pytest
        sys.exit(pytest.main(["-q", "-x", "-p", "no:cacheprovider", *%r]))
    """) % (ROOT, str(tmp_path), str(tmp_path), pins)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, (name, r.returncode, r.stdout[-3000:], r.stderr[-2000:])
