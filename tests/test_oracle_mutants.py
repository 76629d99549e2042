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
    ("non-strict acceptance", "int accept = u[i] * qx < p[x];", "int accept = u[i] * qx <= p[x];", 1),
    ("ratio inverted", "int accept = u[i] * qx < p[x];", "int accept = u[i] * p[x] < qx;", 1),
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
    ("tree ignores the parent link", "if (par[c - 1] == node &&", "if (", 1),
    ("packed offsets off by one", "cu[b + 1] = cu[b] + accept_len[b];",
     "cu[b + 1] = cu[b] + accept_len[b] + (b == 0);", 1),
    ("token bound off by one", "if (x < 0 || x >= V) return OR_BAD_TOKEN;",
     "if (x < 0 || x > V) return OR_BAD_TOKEN;", 2),
    ("accepted drafts not copied",
     "for (int i = 0; i < n; ++i) tokens[i] = draft_tokens[b * (size_t)K + (size_t)i];\n  tokens[n] = t;",
     "for (int i = 0; i < n; ++i) tokens[i] = 0;\n  tokens[n] = t;", 1),
    ("mask bits read from the top", "(mask_row[j / 32] >> (j % 32)) & 1u",
     "(mask_row[j / 32] >> (31 - j % 32)) & 1u", 1),
    ("mask words indexed by token modulo", "(mask_row[j / 32] >> (j % 32)) & 1u",
     "(mask_row[j % 32 % ((V + 31) / 32)] >> (j % 32)) & 1u", 1),
    ("draft row left unmasked",
     "      apply_token_mask(lrow, V, mask_row_of(mask, K, V, b, i));\n      if (!row_is_valid",
     "      if (!row_is_valid", 1),
    ("bonus row takes the previous position's mask", "mask_row_of(mask, K, V, b, K_b)",
     "mask_row_of(mask, K, V, b, K_b > 0 ? K_b - 1 : 0)", 1),
    ("mask rows strided by K", "return mask + (b * (size_t)(K + 1) + (size_t)i) * words;",
     "return mask + (b * (size_t)K + (size_t)i) * words;", 1),
    ("greedy ignores the mask", "    apply_token_mask(row, V, mask_row_of(mask, K, V, b, i));\n",
     "", 1),
    ("n-gram pattern may match itself", "for (int s = 0; s + n < len && found < 0; ++s) {",
     "for (int s = 0; s + n <= len && found < 0; ++s) {", 1),
    ("n-gram takes the latest occurrence", "if (equal) found = s;",
     "if (equal) { found = s; for (int s2 = s + 1; s2 + n < len; ++s2) { int e2 = 1; "
     "for (int t = 0; t < n; ++t) if (c[s2 + t] != pattern[t]) { e2 = 0; break; } "
     "if (e2) found = s2; } }", 1),
    ("n-gram tries the shortest n first",
     "for (int n = n_max; n >= n_min; --n) {\n      if (len < n + 1) continue;",
     "for (int n = n_min; n <= n_max; ++n) {\n      if (len < n + 1) continue;", 1),
    ("top-k drops the class at the cut", "if (l[j] < vk) p[j] = 0.0;", "if (l[j] <= vk) p[j] = 0.0;", 1),
    ("top-p counts the class itself", "if (!dropping && above < top_p) {",
     "if (!dropping && above + mass < top_p) {", 1),
    ("top-p on the unrenormalised top-k",
     "    for (int j = 0; j < V; ++j) p[j] /= Z;\n  }\n  if (!isnan(forced)) {",
     "  }\n  if (!isnan(forced)) {", 1),
    ("draft left unfiltered",
     "      flags[i] |= filter_top_k_top_p(lrow, q, V, top_k, top_p, order,\n"
     "                                     cut ? cut[K + 1 + i] : NAN,\n"
     "                                     cut_margin ? &cut_margin[K + 1 + i] : NULL);\n", "", 1),
    ("bonus row left unfiltered",
     "    flags[K_b] |= filter_top_k_top_p(lrow, p, V, top_k, top_p, order, cut ? cut[K_b] : NAN,\n"
     "                                     cut_margin ? &cut_margin[K_b] : NULL);\n", "", 1),
    ("typical entropy in bits", "if (p[j] > 0) H -= p[j] * log(p[j]);",
     "if (p[j] > 0) H -= p[j] * log2(p[j]);", 1),
    ("typical threshold takes the max", "return t < eps ? t : eps;", "return t > eps ? t : eps;", 1),
    ("typical test not strict", "int pass = p[x] > thr;", "int pass = p[x] >= thr;", 1),
    ("typical draw from the bonus row", "load_row(target, dtype, (size_t)b * (size_t)(K + 1) + (size_t)n, V, l);",
     "load_row(target, dtype, (size_t)b * (size_t)(K + 1) + (size_t)K_b, V, l);", 1),
    ("typical tree keeps the highest id", "if (acc[n] && depth[n] > depth[best]) best = n;",
     "if (acc[n] && depth[n] >= depth[best]) best = n;", 1),
    ("typical tree tests under the node's own row", "double px = pp[(size_t)pa * (size_t)V + (size_t)t];",
     "double px = pp[(size_t)(acc[pa] ? pa : pa) * (size_t)V + (size_t)t] * (n % 2 ? 1.0 : 0.5);", 1),
    ("n-gram drafts start one late", "drafts[(size_t)b * (size_t)K + (size_t)t] = c[found + n + t];",
     "drafts[(size_t)b * (size_t)K + (size_t)t] = c[found + n + t + 1 < len ? found + n + t + 1 : found + n + t];", 1),
    # lossless tree verification by rejection sampling
    ("tree sampler keeps a rejected token in the residual", "          w[x] = 0.0;",
     "          w[x] = w[x];", 1),
    ("tree sampler tests against p instead of the residual",
     "double theta = W > 0 ? w[x] / W : 0.0;", "double theta = p[x];", 1),
    ("tree sampler draws from p", "tokens[len++] = sv_oracle_inverse_cdf(w, V, u[0], &margin);",
     "tokens[len++] = sv_oracle_inverse_cdf(p, V, u[0], &margin);", 1),
    ("tree sampler draws with the node's uniform",
     "tokens[len++] = sv_oracle_inverse_cdf(w, V, u[0], &margin);",
     "tokens[len++] = sv_oracle_inverse_cdf(w, V, u[node], &margin);", 1),
    ("tree sampler tests children in reverse order",
     "for (int c = 1; c <= N && next < 0; ++c) {", "for (int c = N; c >= 1 && next < 0; --c) {", 1),
    ("tree sampler test not strict", "int accept = u[c] < theta;", "int accept = u[c] <= theta;", 1),
    ("tree depth limit off by one", "if (depth[n] > max_depth) return OR_BAD_TREE;",
     "if (depth[n] >= max_depth + (n > 2)) return OR_BAD_TREE;", 1),
    ("a node may be its own parent", "if (pa < 0 || pa >= n) return OR_BAD_TREE;",
     "if (pa < 0 || pa > n) return OR_BAD_TREE;", 1),
    ("per-request trees read the first tree",
     "const int32_t* par = parent + (size_t)b * (size_t)parent_stride;",
     "const int32_t* par = parent;", 3),
    # checking hooks
    ("forced cut distances swapped", "d = forced < own ? front - top_p : top_p - through;",
     "d = forced < own ? top_p - through : front - top_p;", 1),
    ("forced cut drops its own class", "        if (l[j] < forced) p[j] = 0.0;",
     "        if (l[j] <= forced) p[j] = 0.0;", 1),
    ("flip ignored (sampling)", "    if (flip && flip[i]) accept = !accept;\n", "", 1),
    ("flip ignored (typical)",
     "      if (flip && flip[(size_t)b * (size_t)K + (size_t)i]) pass = !pass;\n", "", 1),
    ("flip ignored (typical tree)", "          if (fl && fl[n]) acc[n] = !acc[n];\n", "", 1),
    ("probe step off by one", "    if (j < t) below += w[j];", "    if (j <= t) below += w[j];", 1),
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
