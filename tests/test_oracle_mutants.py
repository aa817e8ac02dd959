"""The oracle's pins catch plausible slips in the oracle.

Each case below plants one mistake in a copy of the oracle — a dropped term, a wrong sign,
a transposed index, swapped operands, read-before-write, a wrong tie-break or ordering, a
slip in the reverse-mode rules — and runs the oracle's pin files (tests/test_oracle_pins.py,
tests/test_oracle_backward_pins.py, tests/test_oracle_project_pins.py) against that copy in
a subprocess: at least one pin has to fail.  The unmodified copy, run the same way, has to
pass.  Mistakes in the C++ part are planted in a copy of oracle/sdm_oracle.cpp compiled to a
library of its own; mistakes in the Python part are planted in the module's source before it
is executed.  The oracle in the repository is never modified; every planted mistake keeps
all memory accesses in bounds.

Equations the pins hold the oracle to: "Sparse Delta Memory (SDM)" technical summary,
gist.science/it/paper/2607.07386, section "Meccanismo Core", items 1-4.
"""
import concurrent.futures
import json
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PIN_FILES = ["tests/test_oracle_pins.py", "tests/test_oracle_backward_pins.py",
             "tests/test_oracle_project_pins.py"]


def _swap_read_and_write(src: str) -> str:
    """Token loop of the forward scan with the read (item 4) before the write (item 3)."""
    i3 = src.index("    // item 3: gated delta update")
    i4 = src.index("    // item 4: weighted read")
    end_marker = "    }\n  }\n}\n\n// Softmax backward"
    i_end = src.index(end_marker, i4) + len("    }\n")
    write, read = src[i3:i4], src[i4:i_end]
    return src[:i3] + read + write + src[i_end:]


# (name, part, [(old, new), ...] or a callable on the source text)
MUTANTS = [
    # selection ("Meccanismo Core" item 2)
    ("tie-break by higher index", "cpp", [("return a.i < b.i;", "return a.i > b.i;")]),
    ("lowest scores first", "cpp", [("if (a.v != b.v) return a.v > b.v;", "if (a.v != b.v) return a.v < b.v;")]),
    ("flat index transposed", "cpp", [("a[p].i * S + b[q].i", "b[q].i * S + a[p].i")]),
    ("both inner lists from half 0", "cpp", [("top_of_half(half1, S, kk, b);", "top_of_half(half0, S, kk, b);")]),
    ("pair sum drops the second half", "cpp", [("const float s = a[p].v + b[q].v;", "const float s = a[p].v;")]),
    ("pair sum with a minus", "cpp", [("const float s = a[p].v + b[q].v;", "const float s = a[p].v - b[q].v;")]),
    # write (item 3)
    ("forget gate dropped", "cpp", [("const double mt = a * row[c];                     // forget gate",
                                     "const double mt = row[c];                     // forget gate")]),
    ("delta update with a minus", "cpp", [("row[c] = mt + b * kw[i] * (double(vt[c]) - mt);",
                                           "row[c] = mt - b * kw[i] * (double(vt[c]) - mt);")]),
    ("error term from the ungated row", "cpp", [("row[c] = mt + b * kw[i] * (double(vt[c]) - mt);",
                                                 "row[c] = mt + b * kw[i] * (double(vt[c]) - row[c]);")]),
    ("write weight dropped", "cpp", [("row[c] = mt + b * kw[i] * (double(vt[c]) - mt);",
                                      "row[c] = mt + b * (double(vt[c]) - mt);")]),
    ("alpha and beta swapped", "cpp", [("    softmax64(sc_w + size_t(t) * W, W, kw.data());\n"
                                        "    const double a = alpha[t], b = beta[t];",
                                        "    softmax64(sc_w + size_t(t) * W, W, kw.data());\n"
                                        "    const double a = beta[t], b = alpha[t];")]),
    ("v of the previous token", "cpp", [("    const float* vt = v + size_t(t) * dv;\n    for (int i = 0; i < W; ++i) {\n"
                                         "      double* row = M + size_t(",
                                         "    const float* vt = v + size_t(t > 0 ? t - 1 : 0) * dv;\n"
                                         "    for (int i = 0; i < W; ++i) {\n      double* row = M + size_t(")]),
    ("softmax exponent negated", "cpp", [("w[i] = std::exp(double(s[i]) - mx);", "w[i] = std::exp(mx - double(s[i]));")]),
    # read (item 4)
    ("read weights uniform", "cpp", [("for (int c = 0; c < dv; ++c) ot[c] += rw[i] * row[c];",
                                      "for (int c = 0; c < dv; ++c) ot[c] += row[c] / R;")]),
    ("read from the write slots", "cpp", [("const double* row = M + size_t(idx_r[size_t(t) * R + i]) * dv;",
                                           "const double* row = M + size_t(idx_w[size_t(t) * W + (i % W)]) * dv;")]),
    ("read before the write", "cpp", _swap_read_and_write),
    # reverse mode of the scan
    ("dalpha without the (1 - b k) factor", "cpp", [("sa += (1.0 - b * k[i]) * gm;", "sa += gm;")]),
    ("dbeta without the write weight", "cpp", [("sb += k[i] * ge;", "sb += ge;")]),
    ("dk without beta", "cpp", [("dk[i] = b * ge;", "dk[i] = ge;")]),
    ("dv without beta", "cpp", [("dvt[c] += b * k[i] * g[c];", "dvt[c] += k[i] * g[c];")]),
    ("state adjoint keeps the delta term", "cpp", [("for (int c = 0; c < dv; ++c) g[c] *= a * (1.0 - b * k[i]);",
                                                    "for (int c = 0; c < dv; ++c) g[c] *= a;")]),
    ("read adjoint without the read weight", "cpp", [("for (int c = 0; c < dv; ++c) g[c] += r[j] * dot[c];",
                                                      "for (int c = 0; c < dv; ++c) g[c] += dot[c];")]),
    ("softmax backward without the centring", "cpp", [("ds[i] = w[i] * (dw[i] - dot);", "ds[i] = w[i] * dw[i];")]),
    # Python part: composition, selection gradient, projections
    ("read slots selected on k'", "py", [("idx_r, sc_r = select(qp, R, n_threads)", "idx_r, sc_r = select(kp, R, n_threads)")]),
    ("selection gradient to the wrong halves", "py", [("np.add.at(out[:, 0], (rows, flat_i // S), flat_d)",
                                                       "np.add.at(out[:, 0], (rows, flat_i % S), flat_d)"),
                                                      ("np.add.at(out[:, 1], (rows, flat_i % S), flat_d)",
                                                       "np.add.at(out[:, 1], (rows, flat_i // S), flat_d)")]),
    ("k' and q' swapped", "py", [("        return a[0], a[1]", "        return a[1], a[0]")]),
    ("head and half axes transposed", "py", [("a = a.reshape(lead + (2, H, 2, S))", "a = a.reshape(lead + (2, 2, H, S))")]),
]

BOOT = """
import json, sys
sys.path.insert(0, {root!r})
import oracle
spec = json.loads(sys.argv[1])
if spec["py"]:
    src = open(oracle.__file__).read()
    for old, new in spec["py"]:
        if src.count(old) != 1:
            sys.exit(3)          # the planted change no longer applies
        src = src.replace(old, new)
    exec(compile(src, oracle.__file__, "exec"), oracle.__dict__)
oracle._lib = oracle.open_library(spec["so"])
import pytest
sys.exit(pytest.main(["-x", "-q", "-p", "no:cacheprovider"] + spec["files"]))
"""


def _plant_cpp(src: str, change) -> str:
    if callable(change):
        out = change(src)
    else:
        out = src
        for old, new in change:
            assert out.count(old) == 1, f"expected one occurrence of {old!r}"
            out = out.replace(old, new)
    assert out != src
    return out


def _run_pins(so: str, py_changes, tmp_path, tag: str) -> subprocess.CompletedProcess:
    spec = json.dumps({"so": so, "py": py_changes, "files": PIN_FILES})
    return subprocess.run([sys.executable, "-c", BOOT.format(root=ROOT), spec], cwd=ROOT,
                          capture_output=True, text=True, timeout=300)


@pytest.fixture(scope="module")
def planted(tmp_path_factory):
    """Every planted case compiled (C++) or prepared (Python), then run against the pins."""
    tmp = tmp_path_factory.mktemp("oracle_mutants")
    with open(oracle._SRC) as f:
        src = f.read()
    clean_so = oracle.build()
    jobs = []
    for n, (name, part, change) in enumerate(MUTANTS):
        if part == "cpp":
            path = tmp / f"mutant{n}.cpp"
            path.write_text(_plant_cpp(src, change))
            jobs.append((name, str(path), str(tmp / f"libmutant{n}.so"), []))
        else:
            jobs.append((name, None, clean_so, [list(c) for c in change]))

    def one(job):
        name, cpp, so, py = job
        if cpp:
            oracle.compile_library(cpp, so)
        return name, _run_pins(so, py, tmp, name)

    workers = max(1, min(8, os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        results = dict(ex.map(one, jobs))
        control = ex.submit(_run_pins, clean_so, [], tmp, "control").result()
    return results, control


def test_unmodified_oracle_passes_through_the_same_harness(planted):
    _, control = planted
    assert control.returncode == 0, control.stdout[-2000:] + control.stderr[-2000:]


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(planted, name):
    results, _ = planted
    r = results[name]
    # exit code 1 with a failed pin (not a crash, a collection error or a change that no
    # longer applies)
    assert r.returncode == 1 and " failed" in r.stdout, \
        f"{name}: pins exit {r.returncode}\n{r.stdout[-2000:]}\n{r.stderr[-2000:]}"
