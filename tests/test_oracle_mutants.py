"""Every plausible mistake in the oracle is caught by one of its pins.

Each case below edits one expression in a private copy of the oracle's C
source (a dropped clamp, a wrong row, a flipped comparison, ...), builds
it, and runs the pin checks of oracle_checks.py against it: at least one
check must fail.  The committed oracle is never modified."""
import ctypes
import os
import subprocess

import pytest

import oracle
import oracle_checks as oc

SRC = os.path.join(os.path.dirname(oracle.__file__), "spec_oracle.c")

MUTANTS = [
    ("residual clamp dropped", "w[j] = r > 0 ? r : 0.0;", "w[j] = r;", 1),
    ("non-strict acceptance", "if (!(u[i] * qx < p[x])) {", "if (!(u[i] * qx <= p[x])) {", 1),
    ("ratio inverted", "if (!(u[i] * qx < p[x])) {", "if (!(u[i] * p[x] < qx)) {", 1),
    ("bonus from the previous row",
     "load_row(target, dtype, b * (size_t)(K + 1) + (size_t)K_b, V, lrow);",
     "load_row(target, dtype, b * (size_t)(K + 1) + (size_t)(K_b > 0 ? K_b - 1 : 0), V, lrow);", 1),
    ("one-hot residual keeps the draft", "double qj = draft ? q[j] : (j == x ? 1.0 : 0.0);",
     "double qj = draft ? q[j] : 0.0;", 1),
    ("draft distribution not tempered", "sv_oracle_tempered_softmax(lrow, V, T, q);",
     "sv_oracle_tempered_softmax(lrow, V, 1.0, q);", 1),
    ("temperature multiplies", "l[j] / T", "l[j] * T", 2),
    ("softmax without the max shift", "p[j] = exp(l[j] / T - M);", "p[j] = exp(l[j] / T);", 1),
    ("argmax keeps the last tie", "if (l[j] > l[best]) best = j;", "if (l[j] >= l[best]) best = j;", 1),
    ("CDF step taken at equality", "if (C > target) {", "if (C >= target) {", 1),
    ("draw uses the position's uniform", "sv_oracle_inverse_cdf(w, V, u[K], &margin);",
     "sv_oracle_inverse_cdf(w, V, u[n], &margin);", 1),
    ("greedy emits the draft at a mismatch", "      n = i;\n      emitted = a;",
     "      n = i;\n      emitted = x;", 1),
    ("tree ignores the parent link", "if (parent[c - 1] == node &&", "if (", 1),
    ("packed offsets off by one", "cu[b + 1] = cu[b] + accept_len[b];",
     "cu[b + 1] = cu[b] + accept_len[b] + (b == 0);", 1),
    ("token bound off by one", "if (x < 0 || x >= V) return OR_BAD_TOKEN;",
     "if (x < 0 || x > V) return OR_BAD_TOKEN;", 2),
    ("accepted drafts not copied",
     "for (int i = 0; i < n; ++i) tokens[i] = draft_tokens[b * (size_t)K + (size_t)i];\n  tokens[n] = t;",
     "for (int i = 0; i < n; ++i) tokens[i] = 0;\n  tokens[n] = t;", 1),
]

FAST_CHECKS = [c for c in oc.ALL_CHECKS] + [
    lambda: oc.check_exact_dense(V=4, K=2, T=0.7, seed=21),
    lambda: oc.check_exact_onehot(V=4, K=2, T=0.9, seed=22),
]


@pytest.mark.parametrize("name,old,new,count", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, count):
    src = open(SRC).read()
    assert src.count(old) == count, "mutation site moved: %r" % old
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", str(so), str(mutant_c), "-lm"], check=True)
    saved = oracle._load()
    oracle._lib = oracle.configure(ctypes.CDLL(str(so)))
    caught = None
    try:
        for check in FAST_CHECKS:
            try:
                check()
            except (AssertionError, ValueError) as e:  # noqa: PERF203
                caught = (getattr(check, "__name__", "check"), str(e)[:200])
                break
    finally:
        oracle._lib = saved
    assert caught is not None, "mutant '%s' passed every pin" % name
