"""Mutation check of the oracle's pins (no GPU).

Each case copies the oracle (``oracle/__init__.py`` and ``oracle/rsa_oracle.c``)
into a temporary folder, plants one plausible mistake in the copy, and reruns
the pin tests (test_oracle_pins.py, test_oracle_ring.py) against it in a
subprocess.  A pin suite that still passes with the mistake in place would not
protect the oracle from it, so every case must make at least one pin fail.
Mistakes are planted in the oracle only, on the CPU, and none of them reads
outside its arrays."""
import concurrent.futures
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle")
PINS = [os.path.join(ROOT, "tests", "test_oracle_pins.py"), os.path.join(ROOT, "tests", "test_oracle_ring.py")]

C = "rsa_oracle.c"
PY = "__init__.py"

# (name, file, [(text, replacement), ...]); each text must occur exactly once.
MUTANTS = [
    ("exclusive causal mask", C, [("if (causal && t + 1 < hi)\n                hi = t + 1;",
                                  "if (causal && t < hi)\n                hi = t;")]),
    ("mask admits one future key", C, [("if (causal && t + 1 < hi)\n                hi = t + 1;",
                                       "if (causal && t + 2 < hi)\n                hi = t + 2;")]),
    ("scale 1/d instead of 1/sqrt(d)", C, [("1.0 / sqrt((double)d)", "1.0 / (double)d")]),
    ("no score scale", C, [("1.0 / sqrt((double)d)", "1.0")]),
    ("K and V swapped", C, [("dot += q[x] * load_elem(k, dtype", "dot += q[x] * load_elem(v, dtype"),
                            ("o[x] += p * load_elem(v, dtype", "o[x] += p * load_elem(k, dtype")]),
    ("lse without the max", C, [("lse[r] = m + log(l);", "lse[r] = log(l);")]),
    ("natural-log lse taken in base 2", C, [("lse[r] = m + log(l);", "lse[r] = m + log2(l);")]),
    ("head stride transposed", C, [("const int64_t head = (b * H + h) * T;",
                                    "const int64_t head = (h * B + b) * T;")]),
    ("probabilities not normalised", C, [("const double p = exp(s[j - kv_lo] - m) / l;",
                                          "const double p = exp(s[j - kv_lo] - m);")]),
    ("normaliser without the max shift", C, [("l += exp(s[j - kv_lo] - m);", "l += exp(s[j - kv_lo]);")]),
    ("bf16 widened from the wrong bits", C, [("<< 16;", "<< 15;")]),
    ("kv offset of a pair ignored", PY, [("out, lse = _attend_tagged(q_rows, tq, k, v, rows, causal, kv_off, "
                                          "kv_off + kv_len, nthreads)",
                                          "out, lse = _attend_tagged(q_rows, tq, k, v, rows, causal, 0, "
                                          "kv_len, nthreads)")]),
    ("merge weight sign flipped", PY, [("wb = np.where(finite, np.exp(lse_b - Ms), 0.0)",
                                        "wb = np.where(finite, np.exp(Ms - lse_b), 0.0)")]),
    ("ring turns the wrong way", PY, [("        j = (i - r) % N\n        if causal and j > i:",
                                       "        j = (i + r) % N\n        if causal and j > i:")]),
    ("causal ring drops the diagonal", PY, [("        if causal and j > i:\n            continue\n        pairs.append",
                                             "        if causal and j >= i:\n            continue\n        pairs.append")]),
    ("chunk ranges shifted by one", PY, [("    return i * Tc, (i + 1) * Tc", "    return i * Tc + 1, (i + 1) * Tc + 1")]),
    ("two-pass rows not normalised", PY, [("        P = E / Z\n", "        P = E\n")]),
    ("(m, l, o) merge drops the rescale of l", PY, [("    l_new = l_a * sa + l_b * sb", "    l_new = l_a + l_b")]),
    ("useful FLOPs count T^2/2 pairs", PY, [("    pairs = T * (T + 1) // 2 if causal else T * T\n    return 4.0 * B * H * d * pairs",
                                            "    pairs = T * T // 2 if causal else T * T\n    return 4.0 * B * H * d * pairs")]),
]


def _make_mutant(tmp, fname, edits):
    pkg = os.path.join(tmp, "oracle")
    os.makedirs(pkg)
    for f in (C, PY):
        shutil.copy(os.path.join(ORACLE, f), os.path.join(pkg, f))
    path = os.path.join(pkg, fname)
    with open(path) as fh:
        src = fh.read()
    for old, new in edits:
        assert src.count(old) == 1, f"mutation site not found exactly once in {fname}: {old!r}"
        src = src.replace(old, new)
    with open(path, "w") as fh:
        fh.write(src)
    return tmp


def _run_pins(folder):
    env = dict(os.environ, RSA_ORACLE_UNDER_TEST=folder, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider", *PINS]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, (r.stdout + r.stderr)[-2000:]


def test_unmutated_copy_passes_every_pin(tmp_path):
    # the harness itself: an unchanged copy of the oracle must pass
    rc, out = _run_pins(_make_mutant(str(tmp_path), PY, []))
    assert rc == 0, out


def test_every_planted_mistake_fails_a_pin(tmp_path):
    folders = {}
    for i, (name, fname, edits) in enumerate(MUTANTS):
        folders[name] = _make_mutant(str(tmp_path / f"m{i}"), fname, edits)
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
        results = dict(zip(folders, ex.map(_run_pins, folders.values())))
    survived = [name for name, (rc, _) in results.items() if rc == 0]
    assert not survived, f"mistakes no pin catches: {survived}"
    # a failing run must come from a failing pin, not from a broken build
    for name, (rc, out) in results.items():
        assert rc == 1, f"{name}: pytest exited {rc}:\n{out}"
