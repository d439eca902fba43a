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
    "greedy chain accepts every draft": [("      ok = (st.argmax == d);", "      ok = true;")],
    "chain draft outside the vocabulary not flagged": [
        ("    if (d < 0 || d >= a.lg.vocab) {\n      rr.status |= kTokenRange;\n",
         "    if (d < 0 || d >= a.lg.vocab) {\n"),
    ],
    "chain tested rows with NaN or +inf not flagged": [
        ("    RowDist st = row_dist(a.lg, row, T);\n    if (st.nonfinite) rr.status |= kNonFinite;\n    if (st.argmax < 0) {\n      how = kUnusable;",
         "    RowDist st = row_dist(a.lg, row, T);\n    if (st.argmax < 0) {\n      how = kUnusable;"),
    ],
    "greedy chain bonus from the first row": [
        ("  if (greedy) {\n    rr.bonus = static_cast<int32_t>(st.argmax);\n    return rr;",
         "  if (greedy) {\n    rr.bonus = static_cast<int32_t>(row_dist(a.lg, start, 0.0).argmax);\n    return rr;"),
    ],
    "greedy tree stop token is a child's token": [
        ("      if (next < 0) {\n        rr.bonus = static_cast<int32_t>(st.argmax);",
         "      if (next < 0) {\n        rr.bonus = kids.empty() ? static_cast<int32_t>(st.argmax) : tok[kids[0]];"),
    ],
    "commit offsets count the accepted drafts only": [
        ("o.commit_cu[b + 1] = o.commit_cu[b] + o.num_out[b];", "o.commit_cu[b + 1] = o.commit_cu[b] + o.num_out[b] - 1;"),
    ],
    "draw gap not normalised by the total weight": [
        ("const double lower = prev > 0.0 ? (t - prev) / S : kInf;", "const double lower = prev > 0.0 ? (t - prev) : kInf;"),
    ],
    "target-only gap ignores the single-token threshold": [
        ("std::min(std::fabs(u - c / a.th_acc), std::fabs(pk - a.th_single))", "std::fabs(u - c / a.th_acc)"),
    ],
    "destination position one past the committed offset": [
        ("o.commit_dst_pos[dst] = seq_lens[b] + k;", "o.commit_dst_pos[dst] = seq_lens[b] + k + 1;"),
    ],
}


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
    "sample-then-match draws every row with the first row's uniform": (
        "match.py", [("t, g = oracle.sample_index(p, float(w.u_accept[row]))",
                      "t, g = oracle.sample_index(p, float(w.u_accept[start]))")],
        ["tests/test_match_oracle.py"]),
    "sample-then-match emits the draft instead of its own draw at a mismatch": (
        "match.py", [("            if d != t:\n                s, tok = j, int(t)",
                      "            if d != t:\n                s, tok = j, d")],
        ["tests/test_match_oracle.py"]),
    "sample-then-match draws from the argmax row at temperature 1": (
        "match.py", [("p = oracle.row_probs(w.logits, w.dtype, row, T)", "p = oracle.row_probs(w.logits, w.dtype, row, 1.0)")],
        ["tests/test_match_oracle.py"]),
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
    "parity rule lets a close test exempt the prefix before it": (
        "parity.py", [("            k0 = int(close[0])", "            k0 = 0")], ["tests/test_parity_rule.py"]),
    "parity rule skips the validity check of a flagged request": (
        "parity.py", [("        for msg in _path_valid(w, b, g):", "        for msg in []:")], ["tests/test_parity_rule.py"]),
    "parity rule compares no commit lists once a request is flagged": (
        "parity.py", [("        bad.extend(_commit_lists_ok(w, g))", "        pass")], ["tests/test_parity_rule.py"]),
    "parity rule exempts every acceptance test": (
        "parity.py", [("close = np.nonzero(test_gap[b] < tol)[0]", "close = np.nonzero(test_gap[b] < 1.0)[0]")],
        ["tests/test_parity_rule.py"]),
}




def _planted_source(name):
    src = open(SRC).read()
    for old, new in MUTATIONS[name]:
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new)
    return src


def _run_pins(sys_path, lib, pins):
    """Run the pin files in a child process with `sys_path` first on its path (and, for a planted oracle.cpp,
    its library in place of the oracle's own).  Returns (exit status, output tail)."""
    setup = "oracle._LIB = %r\noracle.build = lambda force=False: %r\n" % (lib, lib) if lib else ""
    code = textwrap.dedent("""
        import sys
        for p in %r:
            sys.path.insert(0, p)
        import oracle, oracle.dspark, oracle.match, oracle.tree_build, oracle.parity
    """) % (sys_path,) + setup + textwrap.dedent("""
        import pytest
        sys.exit(pytest.main(["-q", "-x", "-p", "no:cacheprovider", *%r]))
    """) % (pins,)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-3000:] + r.stderr[-2000:]


def _cpp_case(name, d):
    cpp = d / "oracle_planted.cpp"
    cpp.write_text(_planted_source(name))
    lib = str(d / "liboracle_planted.so")
    r = subprocess.run(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", str(cpp), "-o", lib],
                       capture_output=True, text=True)
    if r.returncode != 0:
        return -1000, r.stderr[-2000:]
    return _run_pins([ROOT], lib, PINS)


def _py_case(name, d):
    fname, edits, pins = PY_MUTATIONS[name]
    pkg = d / "oracle"
    shutil.copytree(os.path.join(ROOT, "oracle"), pkg, ignore=shutil.ignore_patterns("*.tmp*", "__pycache__"))
    path = pkg / fname
    src = path.read_text()
    for old, new in edits:
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new)
    path.write_text(src)
    return _run_pins([ROOT, str(d)], None, pins)


@pytest.fixture(scope="module")
def planted(tmp_path_factory):
    """Every planted case, built and run against the pins concurrently: (kind, name) -> (exit status, output)."""
    from concurrent.futures import ThreadPoolExecutor
    import oracle
    oracle.build()  # the Python cases copy the oracle with its library already built
    cases = [("cpp", n) for n in sorted(MUTATIONS)] + [("py", n) for n in sorted(PY_MUTATIONS)]

    def run(case):
        kind, name = case
        d = tmp_path_factory.mktemp("planted")
        return (_cpp_case if kind == "cpp" else _py_case)(name, d)

    with ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        return dict(zip(cases, ex.map(run, cases)))


# exit status 1: the pins ran and one failed (0 would mean every pin passed; anything else a crash or an error)
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_fail_on_a_planted_mistake(name, planted):
    rc, out = planted[("cpp", name)]
    assert rc == 1, (name, rc, out)


@pytest.mark.parametrize("name", sorted(PY_MUTATIONS))
def test_python_oracle_pins_fail_on_a_planted_mistake(name, planted):
    rc, out = planted[("py", name)]
    assert rc == 1, (name, rc, out)
