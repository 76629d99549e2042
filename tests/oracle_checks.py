"""Checks that pin the fp64 oracle to facts outside itself.

Each ``check_*`` function raises AssertionError on a mismatch.  The pytest
wrappers live in test_oracle_pins.py; test_oracle_mutants.py runs the same
checks against deliberately broken copies of the oracle to show that every
plausible mistake is caught by at least one of them.

What pins what:
  * library routines: scipy's softmax, numpy's argmax (first maximum) and
    searchsorted over a cumulative sum (smallest j with C_j > u*W);
  * hand-derived worked examples under tests/golden/ (closed forms);
  * the exactness theorem of rejection sampling ("推测解码与 MTP" (juejin.cn),
    the "正确性保证" part of §2): the token emitted at each position is
    distributed exactly as the target distribution there.  Measured by
    treating the oracle as a black box and locating, by bisection over the
    uniforms, the exact u-intervals that lead to each outcome;
  * a chi-square test over 10^6 seeded draws;
  * invariants: 1 <= accept_len <= K+1 (§2.3 of the same page), all
    accepted => K+1 tokens, q == p => everything accepted, one-hot drafts
    accepted exactly when u < p(x), zero-probability drafts never accepted;
  * the T -> 0 limit of sampling equals greedy verification;
  * tree verification against a brute-force enumeration of root paths.
"""
from __future__ import annotations

import json
import os

import numpy as np
import scipy.special
import scipy.stats

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _f(v):
    if isinstance(v, str):
        return {"-inf": -np.inf, "inf": np.inf, "nan": np.nan}[v]
    return float(v)


def _rows(rows):
    return np.asarray([[_f(v) for v in r] for r in rows], dtype=np.float32)


# ---------------------------------------------------------------------------
# library pins
# ---------------------------------------------------------------------------

def check_softmax_matches_scipy():
    rng = np.random.default_rng(101)
    for V in (1, 2, 7, 1000, 32000):
        for T in (0.05, 0.8, 1.0, 2.0):
            l = rng.standard_normal(V) * 3.0
            if V > 2:
                l[rng.random(V) < 0.1] = -np.inf
                l[0] = 0.5
            got = oracle.tempered_softmax(l, T)
            ref = scipy.special.softmax(l / T)
            np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-300)
    # far from zero: exp() stays in range only because of the max shift
    l = np.array([1000.0, 999.0, 998.5, -1e4])
    np.testing.assert_allclose(oracle.tempered_softmax(l, 0.7),
                               scipy.special.softmax(l / 0.7), rtol=1e-12)


def check_argmax_matches_numpy():
    rng = np.random.default_rng(102)
    for V in (1, 2, 3, 17, 1000):
        for _ in range(20):
            l = rng.integers(-3, 4, size=V).astype(np.float64)  # many exact ties
            assert oracle.argmax(l) == int(np.argmax(l)), (l, oracle.argmax(l))
    l = np.array([-0.0, 0.0, -1.0])
    assert oracle.argmax(l) == 0
    l = np.array([-np.inf, -5.0, 2.0, 2.0, -np.inf])
    assert oracle.argmax(l) == 2


def _searchsorted_draw(w, u):
    c = np.cumsum(w)
    j = int(np.searchsorted(c, u * c[-1], side="right"))
    if j >= len(w):
        j = int(np.nonzero(w > 0)[0][-1])
    return j


def check_inverse_cdf_matches_searchsorted():
    rng = np.random.default_rng(103)
    for V in (1, 2, 5, 64, 5000):
        for _ in range(50):
            w = rng.random(V)
            w[rng.random(V) < 0.3] = 0.0
            if not (w > 0).any():
                w[V // 2] = 1.0
            u = float(rng.random())
            t, _ = oracle.inverse_cdf(w, u)
            assert t == _searchsorted_draw(w, u), (V, u, t)
    # zero-weight tokens are never drawn, not even at u = 0 or with a
    # leading run of zeros
    w = np.array([0.0, 0.0, 0.25, 0.0, 0.75])
    for u in (0.0, 1e-300, 0.2499999, 0.25, 0.9999999):
        t, _ = oracle.inverse_cdf(w, u)
        assert w[t] > 0 and t == _searchsorted_draw(w, u), (u, t)


# ---------------------------------------------------------------------------
# worked examples
# ---------------------------------------------------------------------------

def check_golden_sampling():
    for name in ("verify_dense_v3.json", "verify_onehot_v4.json"):
        g = _golden(name)
        V, K, T = g["V"], g["K"], g["T"]
        target = np.log(np.asarray(g["target_probs"])).astype(np.float32)
        draft = None
        if g["mode"] == "dense":
            draft = np.log(np.asarray(g["draft_probs"])).astype(np.float32)[None]
        for case in g["cases"]:
            out = oracle.sample(target[None], draft, np.asarray([case["draft_tokens"]]),
                                np.asarray([case["uniforms"]], np.float32), T)
            assert out["status"][0] == 0
            assert list(out["tokens"][0]) == case["tokens"], (name, case, out["tokens"][0])
            assert out["accept_len"][0] == case["accept_len"], (name, case)
            np.testing.assert_allclose(out["accept_prob"][0], case["accept_prob"], atol=1e-6)


def check_golden_greedy():
    g = _golden("verify_greedy_ties.json")
    target = _rows(g["target_logits"])[None]
    for case in g["cases"]:
        lens = None if "draft_len" not in case else np.asarray([case["draft_len"]])
        out = oracle.greedy(target, np.asarray([case["draft_tokens"]]), draft_lens=lens)
        assert out["status"][0] == 0
        assert list(out["tokens"][0]) == case["tokens"], (case, out["tokens"][0])
        assert out["accept_len"][0] == case["accept_len"]
        # the sampling entry at temperature 0 is the same rule
        out2 = oracle.sample(target, None, np.asarray([case["draft_tokens"]]),
                             np.zeros((1, g["K"] + 1), np.float32), 0.0, draft_lens=lens)
        assert list(out2["tokens"][0]) == case["tokens"]


def check_golden_tree():
    g = _golden("verify_tree_small.json")
    parent = np.asarray(g["parent"], np.int32)
    for req in g["requests"]:
        target = _rows(req["target_logits"])[None]
        out = oracle.tree(target, parent, np.asarray([g["node_tokens"]]), g["max_depth"])
        assert out["status"][0] == 0
        assert list(out["tokens"][0]) == req["tokens"], (req, out["tokens"][0])
        assert list(out["path"][0]) == req["path"], (req, out["path"][0])
        assert out["accept_len"][0] == req["accept_len"]


def check_golden_compact():
    g = _golden("compact_small.json")
    cu, packed, bid = oracle.compact(np.asarray(g["tokens"]), np.asarray(g["accept_len"]))
    assert list(cu) == g["cu"] and list(packed) == g["packed"] and list(bid) == g["batch_id"]


# ---------------------------------------------------------------------------
# exactness by measure (the oracle as a black box)
# ---------------------------------------------------------------------------

_ONE_MINUS = float(np.nextafter(1.0, 0.0))


def _bisect(pred, iters=64):
    """Boundary b in [0, 1] with pred true on [0, b) and false on [b, 1),
    for a pred that is monotone (true then false)."""
    if not pred(0.0):
        return 0.0
    if pred(_ONE_MINUS):
        return 1.0
    lo, hi = 0.0, _ONE_MINUS
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if mid <= lo or mid >= hi:
            break
        if pred(mid):
            lo = mid
        else:
            hi = mid
    return hi


class _Request:
    """One request evaluated by the oracle for chosen drafts and uniforms."""

    def __init__(self, target, draft, T, mask=None, top_k=0, top_p=1.0):
        self.top_k, self.top_p = top_k, top_p
        self.target = np.ascontiguousarray(target[None], np.float32)
        self.draft = None if draft is None else np.ascontiguousarray(draft[None], np.float32)
        self.mask = None if mask is None else np.ascontiguousarray(mask[None], np.uint32)
        self.K = target.shape[0] - 1
        self.T = T

    def run(self, drafts, u):
        out = oracle.sample(self.target, self.draft, np.asarray([drafts], np.int32),
                            np.asarray([u], np.float64), self.T, token_mask=self.mask,
                            top_k=self.top_k, top_p=self.top_p)
        assert out["status"][0] == 0
        return out["tokens"][0], int(out["accept_len"][0])


def _emission_law(req, drafts, i):
    """Exact law of the token emitted at position i given drafts (with the
    drafts before i accepted through u_j = 0): returns (theta, residual law)
    where theta is the measure of u_i giving acceptance and the residual
    law is the measure of u_K over each token after a rejection at i."""
    K, V = req.K, req.target.shape[2]
    base = [0.0] * (K + 1)

    def accepted(a):
        u = list(base)
        u[i] = a
        _, L = req.run(drafts, u)
        return L > i + 1

    theta = _bisect(accepted) if i < K else 1.0
    law = np.zeros(V)
    if i < K and theta >= 1.0:
        return theta, law
    u_rej = list(base)
    if i < K:
        u_rej[i] = 0.5 * (theta + 1.0) if theta < _ONE_MINUS else _ONE_MINUS

    def token(s):
        u = list(u_rej)
        u[K] = s
        toks, L = req.run(drafts, u)
        assert L == i + 1
        return int(toks[i])

    prev = 0.0
    for t in range(V):
        edge = 1.0 if t == V - 1 else _bisect(lambda s: token(s) <= t)
        law[t] = edge - prev
        prev = edge
    return theta, law


def check_exact_dense(V=5, K=3, T=0.8, seed=0, mask=False):
    """P(y_i = t | drafts before i accepted) = p_i(t) with x_i ~ q_i, for
    every position including the bonus, to 1e-12."""
    rng = np.random.default_rng(seed)
    l = (rng.standard_normal((K + 1, V)) * 1.3).astype(np.float32)
    d = (l[:K] + rng.standard_normal((K, V)) * 0.9).astype(np.float32)
    if mask:
        l[0, 1] = -np.inf          # a token the target rules out
        d[min(1, K - 1), 2] = -np.inf  # a token the draft never proposes
    req = _Request(l, d, T)
    p = scipy.special.softmax(l.astype(np.float64) / T, axis=-1)
    q = scipy.special.softmax(d.astype(np.float64) / T, axis=-1)
    prefix = [int(np.argmax(p[j] * q[j])) for j in range(K)]  # p > 0 and q > 0
    for i in range(K + 1):
        emitted = np.zeros(V)
        xs = range(V) if i < K else [0]
        for x in xs:
            if i < K and q[i, x] == 0:
                continue
            drafts = prefix[:i] + [x] + prefix[i + 1:] if i < K else list(prefix)
            theta, law = _emission_law(req, drafts, i)
            if i < K:
                emitted[x] += q[i, x] * theta
                emitted += q[i, x] * (1.0 - theta) * law
            else:
                emitted = law
        np.testing.assert_allclose(emitted, p[i], rtol=0, atol=1e-12,
                                   err_msg="position %d" % i)


def check_exact_onehot(V=5, K=2, T=1.3, seed=1):
    """Deterministic proposer: for every proposed x, P(y_i = t) = p_i(t);
    acceptance has measure p_i(x) and the residual never emits x."""
    rng = np.random.default_rng(seed)
    l = (rng.standard_normal((K + 1, V)) * 1.5).astype(np.float32)
    req = _Request(l, None, T)
    p = scipy.special.softmax(l.astype(np.float64) / T, axis=-1)
    prefix = [int(np.argmax(p[j])) for j in range(K)]
    for i in range(K + 1):
        for x in (range(V) if i < K else [0]):
            drafts = prefix[:i] + [x] + prefix[i + 1:] if i < K else list(prefix)
            theta, law = _emission_law(req, drafts, i)
            if i < K:
                assert abs(theta - min(1.0, p[i, x])) < 1e-12, (i, x, theta, p[i, x])
                assert law[x] == 0.0, "residual emitted the rejected draft"
                emitted = (1.0 - theta) * law
                emitted[x] += theta
            else:
                emitted = law
            np.testing.assert_allclose(emitted, p[i], rtol=0, atol=1e-12,
                                       err_msg="position %d draft %d" % (i, x))


def check_chi_square(B=1_000_000, V=16, K=3, T=0.9, seed=7, threads=8):
    """10^6 seeded draws with drafts sampled from q: the emitted token at
    each position, given the earlier drafts were accepted, follows p_i."""
    rng = np.random.default_rng(seed)
    l = (rng.standard_normal((K + 1, V)) * 1.5).astype(np.float32)
    d = (l[:K] + rng.standard_normal((K, V)) * 0.8).astype(np.float32)
    p = scipy.special.softmax(l.astype(np.float64) / T, axis=-1)
    q = scipy.special.softmax(d.astype(np.float64) / T, axis=-1)
    drafts = np.stack([rng.choice(V, size=B, p=q[i]) for i in range(K)], axis=1).astype(np.int32)
    u = rng.random((B, K + 1))
    target = np.ascontiguousarray(np.broadcast_to(l, (B, K + 1, V)))
    draft = np.ascontiguousarray(np.broadcast_to(d, (B, K, V)))
    out = oracle.sample(target, draft, drafts, u, T, threads=threads)
    L = out["accept_len"]
    assert (out["status"] == 0).all()
    for i in range(K + 1):
        sel = L >= i + 1
        obs = np.bincount(out["tokens"][sel, i], minlength=V)
        exp = p[i] * sel.sum()
        pval = scipy.stats.chisquare(obs, exp).pvalue
        assert pval > 1e-3, "position %d: chi-square p-value %.3g" % (i, pval)


# ---------------------------------------------------------------------------
# invariants and limits
# ---------------------------------------------------------------------------

def check_invariants(seed=11):
    rng = np.random.default_rng(seed)
    B, K, V, T = 400, 4, 50, 1.1
    l = (rng.standard_normal((B, K + 1, V)) * 2).astype(np.float32)
    d = (l[:, :K] + rng.standard_normal((B, K, V))).astype(np.float32)
    drafts = rng.integers(0, V, size=(B, K)).astype(np.int32)
    lens = rng.integers(0, K + 1, size=B).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    for dr in (d, None):
        out = oracle.sample(l, dr, drafts, u, T, draft_lens=lens)
        L = out["accept_len"]
        assert (out["status"] == 0).all()
        assert ((L >= 1) & (L <= lens + 1)).all()
        for b in range(B):
            toks = out["tokens"][b]
            assert (toks[:L[b]] >= 0).all() and (toks[L[b]:] == -1).all()
            assert (toks[:L[b] - 1] == drafts[b, :L[b] - 1]).all()
            if L[b] == lens[b] + 1:
                assert (toks >= 0).sum() == lens[b] + 1
    # q == p (draft logits equal to the target logits): always accepted
    out = oracle.sample(l, np.ascontiguousarray(l[:, :K]), drafts, u, T)
    assert (out["accept_len"] == K + 1).all()
    np.testing.assert_array_equal(out["accept_prob"], 1.0)


def check_onehot_accept_iff_u_below_p(seed=12):
    rng = np.random.default_rng(seed)
    B, V, T = 2000, 30, 0.7
    l = (rng.standard_normal((B, 2, V)) * 2).astype(np.float32)
    drafts = rng.integers(0, V, size=(B, 1)).astype(np.int32)
    u = rng.random((B, 2)).astype(np.float32)
    out = oracle.sample(l, None, drafts, u, T)
    px = scipy.special.softmax(l[:, 0].astype(np.float64) / T, axis=-1)[np.arange(B), drafts[:, 0]]
    clear = np.abs(u[:, 0] - px) > 1e-9
    acc = out["accept_len"] == 2
    assert (acc[clear] == (u[clear, 0] < px[clear])).all()
    np.testing.assert_allclose(out["accept_prob"][:, 0], px, rtol=1e-12)


def check_zero_probability_draft_rejected():
    """A draft the target rules out (logit -inf, p = 0) is never accepted,
    even with u = 0; nor is it drawn by the residual."""
    l = np.array([[[0.0, -np.inf, 1.0], [0.0, 0.0, 0.0]]], np.float32)
    for draft in (None, np.array([[[0.0, 2.0, 0.0]]], np.float32)):
        out = oracle.sample(l, draft, np.array([[1]]), np.array([[0.0, 0.0]], np.float32), 1.0)
        assert out["accept_len"][0] == 1 and out["tokens"][0, 0] == 0
        out = oracle.sample(l, draft, np.array([[1]]), np.array([[0.0, 0.6]], np.float32), 1.0)
        assert out["accept_len"][0] == 1 and out["tokens"][0, 0] == 2


def check_temperature_to_zero_is_greedy(seed=13):
    rng = np.random.default_rng(seed)
    B, K, V = 300, 3, 40
    l = rng.permuted(np.tile(np.arange(V, dtype=np.float32) * 0.25, (B, K + 1, 1)), axis=2)
    am = np.argmax(l, axis=2)
    drafts = np.where(rng.random((B, K)) < 0.7, am[:, :K], rng.integers(0, V, (B, K)))
    drafts = drafts.astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32) * 0.98 + 0.01
    g = oracle.greedy(l, drafts)
    s = oracle.sample(l, None, drafts, u, 1e-3)
    np.testing.assert_array_equal(s["tokens"], g["tokens"])
    np.testing.assert_array_equal(s["accept_len"], g["accept_len"])


def check_errors():
    l = np.zeros((3, 3, 4), np.float32)
    l[:, :, 0] = 1.0
    drafts = np.array([[0, 0], [4, 0], [0, -1]], np.int32)
    out = oracle.sample(l, None, drafts, np.zeros((3, 3), np.float32), 1.0)
    assert list(out["status"]) == [0, oracle.BAD_TOKEN, oracle.BAD_TOKEN]
    assert list(out["accept_len"]) == [3, 0, 0]
    assert (out["tokens"][1:] == -1).all()
    for bad in (np.nan, np.inf):
        lb = l[:1].copy()
        lb[0, 0, 2] = bad
        out = oracle.sample(lb, None, drafts[:1], np.zeros((1, 3), np.float32), 1.0)
        assert out["status"][0] == oracle.BAD_LOGITS
        out = oracle.greedy(lb, drafts[:1])
        assert out["status"][0] == oracle.BAD_LOGITS
    lb = l[:1].copy()
    lb[0, 1, :] = -np.inf
    assert oracle.sample(lb, None, drafts[:1], np.zeros((1, 3)), 1.0)["status"][0] == oracle.BAD_LOGITS
    # rows after the first rejection are never needed, so they are not checked
    lb = l[:1].copy()
    lb[0, 2, 1] = np.nan
    out = oracle.sample(lb, None, np.array([[1, 0]]), np.array([[0.9, 0, 0.5]], np.float32), 1.0)
    assert out["status"][0] == 0 and out["accept_len"][0] == 1
    out = oracle.sample(l[:1], None, drafts[:1], np.zeros((1, 3)), 1.0,
                        draft_lens=np.array([3], np.int32))
    assert out["status"][0] == oracle.BAD_DRAFT_LEN and out["accept_len"][0] == 0


# ---------------------------------------------------------------------------
# grammar masks
# ---------------------------------------------------------------------------

def _allowed(mask_words, V):
    """Decode mask words with numpy's little-endian bit unpacking (an
    independent reading of the layout: bit j % 32 of word j // 32)."""
    w = np.ascontiguousarray(mask_words, dtype="<u4")
    bits = np.unpackbits(w.view(np.uint8), axis=-1, bitorder="little")
    return bits[..., :V].astype(bool)


def _probs_table(rows, V):
    out = np.zeros((len(rows), V))
    for r, row in enumerate(rows):
        for j, v in row.items():
            out[r, int(j)] = v
    return out


def check_golden_masked():
    g = _golden("verify_masked_v40.json")
    V, K, T = g["V"], g["K"], g["T"]
    with np.errstate(divide="ignore"):
        target = np.log(_probs_table(g["target_probs"], V)).astype(np.float32)[None]
        draft = np.log(_probs_table(g["draft_probs"], V)).astype(np.float32)[None]
    mask = np.asarray(g["mask_words"], np.uint32)[None]
    for key, dr in (("onehot_cases", None), ("dense_cases", draft)):
        for case in g[key]:
            out = oracle.sample(target, dr, np.asarray([case["draft_tokens"]]),
                                np.asarray([case["uniforms"]], np.float32), T, token_mask=mask)
            assert out["status"][0] == 0
            assert list(out["tokens"][0]) == case["tokens"], (key, case, out["tokens"][0])
            assert out["accept_len"][0] == case["accept_len"], (key, case)
            np.testing.assert_allclose(out["accept_prob"][0], case["accept_prob"], atol=1e-6)
    for case in g["greedy_cases"]:
        out = oracle.greedy(target, np.asarray([case["draft_tokens"]]), token_mask=mask)
        assert out["status"][0] == 0
        assert list(out["tokens"][0]) == case["tokens"], (case, out["tokens"][0])
        assert out["accept_len"][0] == case["accept_len"]


def check_mask_layout(seed=15):
    """Masks spanning three words: the masked argmax and the masked p(x)
    agree with numpy on the bit-unpacked allowed sets, row by row."""
    rng = np.random.default_rng(seed)
    B, K, V, T = 200, 3, 70, 0.9
    l = (rng.standard_normal((B, K + 1, V)) * 2).astype(np.float32)
    mask = rng.integers(0, 2 ** 32, size=(B, K + 1, (V + 31) // 32), dtype=np.uint64)
    mask = mask.astype(np.uint32)
    allowed = _allowed(mask, V)
    mask[~allowed.any(-1)] |= np.uint32(1)  # keep every row usable
    allowed = _allowed(mask, V)
    ml = np.where(allowed, l.astype(np.float64), -np.inf)
    am = np.argmax(ml, axis=2)
    drafts = np.where(rng.random((B, K)) < 0.6, am[:, :K], rng.integers(0, V, (B, K)))
    drafts = drafts.astype(np.int32)
    g = oracle.greedy(l, drafts, token_mask=mask)
    assert (g["status"] == 0).all()
    for b in range(B):
        n = int(g["accept_len"][b]) - 1
        assert (drafts[b, :n] == am[b, :n]).all() and (n == K or drafts[b, n] != am[b, n])
        assert g["tokens"][b, n] == am[b, n]
    # one-hot sampling with every u = 0: all allowed drafts are accepted and
    # accept_prob is the masked p(x); a disallowed draft has p(x) = 0
    p = scipy.special.softmax(ml / T, axis=-1)
    u = np.zeros((B, K + 1), np.float32)
    s = oracle.sample(l, None, drafts, u, T, token_mask=mask)
    for b in range(B):
        n = int(s["accept_len"][b]) - 1
        px = p[b, np.arange(K), drafts[b]]
        np.testing.assert_allclose(s["accept_prob"][b, :n + (n < K)], np.minimum(1, px)[:n + (n < K)],
                                   rtol=1e-12, atol=0)
        ok = np.nonzero(px == 0)[0]
        assert n == (ok[0] if ok.size else K)
        assert allowed[b, n, s["tokens"][b, n]]


def check_exact_masked(V=6, K=2, T=0.8, seed=16):
    """Exactness under grammar masks: with x_i drawn from the masked draft
    distribution, the emitted token at every position follows the masked,
    renormalised target distribution (scipy softmax over the allowed
    tokens), to 1e-12; dense and one-hot drafts."""
    rng = np.random.default_rng(seed)
    l = (rng.standard_normal((K + 1, V)) * 1.3).astype(np.float32)
    d = (l[:K] + rng.standard_normal((K, V)) * 0.9).astype(np.float32)
    allowed = rng.random((K + 1, V)) < 0.6
    allowed[:, 0] = True
    allowed[np.arange(K + 1), np.arange(K + 1) % V] = False  # a different hole per row
    allowed[:, 0] |= ~allowed.any(-1)
    mask = np.zeros((K + 1, (V + 31) // 32), np.uint32)
    for i in range(K + 1):
        for j in np.nonzero(allowed[i])[0]:
            mask[i, j // 32] |= np.uint32(1 << (j % 32))
    p = np.zeros((K + 1, V))
    q = np.zeros((K, V))
    for i in range(K + 1):
        a = allowed[i]
        p[i, a] = scipy.special.softmax(l[i, a].astype(np.float64) / T)
        if i < K:
            q[i, a] = scipy.special.softmax(d[i, a].astype(np.float64) / T)
    # dense drafts: x_i ~ masked q_i, averaged
    req = _Request(l, d, T, mask)
    prefix = [int(np.argmax(p[j] * q[j])) for j in range(K)]
    for i in range(K + 1):
        emitted = np.zeros(V)
        for x in (range(V) if i < K else [0]):
            if i < K and q[i, x] == 0:
                continue
            drafts = prefix[:i] + [x] + prefix[i + 1:] if i < K else list(prefix)
            theta, law = _emission_law(req, drafts, i)
            if i < K:
                emitted[x] += q[i, x] * theta
                emitted += q[i, x] * (1.0 - theta) * law
            else:
                emitted = law
        np.testing.assert_allclose(emitted, p[i], rtol=0, atol=1e-12,
                                   err_msg="dense position %d" % i)
    # one-hot drafts: for every proposed x, allowed or not, the emitted law is p_i
    req = _Request(l, None, T, mask)
    prefix = [int(np.argmax(p[j])) for j in range(K)]
    for i in range(K):
        for x in range(V):
            drafts = prefix[:i] + [x] + prefix[i + 1:]
            theta, law = _emission_law(req, drafts, i)
            assert abs(theta - min(1.0, p[i, x])) < 1e-12, (i, x, theta, p[i, x])
            emitted = (1.0 - theta) * law
            emitted[x] += theta
            np.testing.assert_allclose(emitted, p[i], rtol=0, atol=1e-12,
                                       err_msg="one-hot position %d draft %d" % (i, x))


# ---------------------------------------------------------------------------
# top-k / top-p
# ---------------------------------------------------------------------------

def np_filter(l, T, top_k, top_p):
    """Filtered distribution of one row through numpy: sort for the k-th
    largest logit, unique value classes and cumulative sums for top-p."""
    l = np.asarray(l, np.float64)
    p = scipy.special.softmax(l / T)
    keep = np.ones(l.size, bool)
    if 0 < top_k < l.size:
        keep &= l >= np.sort(l)[::-1][top_k - 1]
    p = np.where(keep, p, 0.0)
    p /= p.sum()
    if top_p < 1.0:
        vals = np.unique(l[keep])[::-1]
        mass = np.array([p[l == v].sum() for v in vals])
        front = np.concatenate([[0.0], np.cumsum(mass)[:-1]])
        keep &= l >= vals[front < top_p].min()
        p = np.where(keep, p, 0.0)
        p /= p.sum()
    return p


def check_golden_topk_topp():
    g = _golden("verify_topk_topp_v6.json")
    target = np.log(np.asarray(g["target_probs"])).astype(np.float32)[None]
    draft = np.log(np.asarray(g["draft_probs"])).astype(np.float32)[None]
    for case in g["cases"]:
        out = oracle.sample(target, draft if case["mode"] == "dense" else None,
                            np.asarray([case["draft_tokens"]]),
                            np.asarray([case["uniforms"]], np.float32), g["T"],
                            top_k=case["top_k"], top_p=case["top_p"])
        assert out["status"][0] == 0
        assert list(out["tokens"][0]) == case["tokens"], (case, out["tokens"][0])
        assert out["accept_len"][0] == case["accept_len"], case
        np.testing.assert_allclose(out["accept_prob"][0], case["accept_prob"], atol=1e-6)
        assert (out["flags"][0] & oracle.FLAG_CUT).sum() == 0


def check_filter_matches_numpy(seed=18):
    """On rows with many exact ties (logits on a 0.5 grid), the oracle's
    filtered p(x) (one-hot acceptance probability) and p/q (dense) agree
    with the numpy filter for every (top_k, top_p) pair."""
    rng = np.random.default_rng(seed)
    B, V, T = 300, 40, 0.9
    l = (np.round(rng.standard_normal((B, 2, V)) * 4) / 2).astype(np.float32)
    d = (np.round(rng.standard_normal((B, 1, V)) * 4) / 2).astype(np.float32)
    x = rng.integers(0, V, size=(B, 1)).astype(np.int32)
    u = np.full((B, 2), 0.5, np.float32)
    for top_k, top_p in ((0, 0.9), (5, 1.0), (3, 0.5), (1, 1.0), (0, 0.3), (12, 0.95)):
        one = oracle.sample(l, None, x, u, T, top_k=top_k, top_p=top_p)
        den = oracle.sample(l, d, x, u, T, top_k=top_k, top_p=top_p)
        for b in range(B):
            p = np_filter(l[b, 0], T, top_k, top_p)
            q = np_filter(d[b, 0], T, top_k, top_p)
            if one["flags"][b, 0] & oracle.FLAG_CUT:
                continue
            assert abs(one["accept_prob"][b, 0] - min(1.0, p[x[b, 0]])) < 1e-12, (b, top_k, top_p)
            px, qx = p[x[b, 0]], q[x[b, 0]]
            want = min(1.0, px / qx) if qx > 0 else (1.0 if px > 0 else 0.0)
            if not den["flags"][b, 0] & oracle.FLAG_CUT:
                assert abs(den["accept_prob"][b, 0] - want) < 1e-12, (b, top_k, top_p)
    # off-switches: top_k = 0 or >= V and top_p = 1 give the unfiltered result
    a = oracle.sample(l, d, x, u, T)
    for k in (0, V, V + 7):
        b2 = oracle.sample(l, d, x, u, T, top_k=k, top_p=1.0)
        assert (a["tokens"] == b2["tokens"]).all()
        np.testing.assert_array_equal(a["accept_prob"], b2["accept_prob"])
    # top_k = 1 with the argmax as the draft: always accepted, and the
    # residual never happens; the bonus is the last row's argmax class
    am = np.argmax(l[:, 0], axis=1).astype(np.int32)[:, None]
    uniq = np.array([(l[b, 0] == l[b, 0].max()).sum() == 1 for b in range(B)])
    one = oracle.sample(l, None, am, np.full((B, 2), 0.999, np.float32), T, top_k=1)
    assert (one["accept_len"][uniq] == 2).all()
    ok = np.array([(l[b, 1] == l[b, 1].max()).sum() == 1 for b in range(B)]) & uniq
    assert (one["tokens"][ok, 1] == np.argmax(l[ok, 1], axis=1)).all()


def check_forced_cut(seed=27):
    """The checking hook for cuts made elsewhere: forcing the rule's own cut
    changes nothing (margin 0); forcing the class above it (one class fewer)
    when top_p lies 3e-6 above the mass in front of the rule's cut class
    reports margin 3e-6 and renormalises p over the classes kept, as the
    numpy filter computes them; a value that is no class of the row, a cut
    below the top-k cut, another cut than the k-th largest for top-k alone,
    or a cut further than 1e-5 from the rule is not admissible (NaN)."""
    rng = np.random.default_rng(seed)
    B, V, T = 120, 40, 0.9
    l = (np.round(rng.standard_normal((B, 2, V)) * 4) / 2).astype(np.float32)
    x = rng.integers(0, V, size=(B, 1)).astype(np.int32)
    u = np.full((B, 2), 0.5, np.float32)
    nan = np.full((B, 2), np.nan)
    seen = 0
    for b in range(B):
        row = l[b, 0].astype(np.float64)
        p = scipy.special.softmax(row / T)
        vals = np.unique(row)[::-1]
        mass = np.array([p[row == v].sum() for v in vals])
        front = np.concatenate([[0.0], np.cumsum(mass)[:-1]])
        j = int(rng.integers(2, min(6, vals.size - 1)))
        top_p = float(front[j] + 3e-6)  # keeps classes 0..j
        if not (mass[j] > 2e-5 and mass[j - 1] > 2e-5):
            continue
        seen += 1

        def forced(c):
            cuts = nan[b:b + 1].copy()
            cuts[0, 0] = c
            return oracle.sample(l[b:b + 1], None, x[b:b + 1], u[b:b + 1], T, top_p=top_p,
                                 cut_logits=cuts)

        plain = oracle.sample(l[b:b + 1], None, x[b:b + 1], u[b:b + 1], T, top_p=top_p)
        own = forced(vals[j])
        assert own["cut_margin"][0, 0] == 0.0
        assert own["accept_prob"][0, 0] == plain["accept_prob"][0, 0]
        assert (own["tokens"] == plain["tokens"]).all()
        fewer = forced(vals[j - 1])
        assert abs(fewer["cut_margin"][0, 0] - 3e-6) < 1e-12, fewer["cut_margin"]
        kept = np.where(row >= vals[j - 1], p, 0.0)
        kept /= kept.sum()
        assert abs(fewer["accept_prob"][0, 0] - min(1.0, kept[x[b, 0]])) < 1e-12
        assert np.isnan(forced(vals[j - 2])["cut_margin"][0, 0])  # two classes fewer: too far
        assert np.isnan(forced(vals[j + 1])["cut_margin"][0, 0])  # one class more: too far
        assert np.isnan(forced(vals[j] + 0.25)["cut_margin"][0, 0])  # no such class
    assert seen > 20, seen
    # with top-k: a cut below the k-th largest value is not admissible; for
    # top-k alone only the k-th largest value itself is
    row = l[0, 0]
    vk = np.sort(row)[::-1][4]
    below = np.unique(row[row < vk])
    for top_p, c, ok in ((0.99, below.max() if below.size else vk - 1, False),
                         (1.0, vk, True), (1.0, np.unique(row[row > vk]).min(), False)):
        cuts = nan[:1].copy()
        cuts[0, 0] = c
        out = oracle.sample(l[:1], None, x[:1], u[:1], T, top_k=5, top_p=top_p, cut_logits=cuts)
        assert (out["cut_margin"][0, 0] == 0.0) if ok else np.isnan(out["cut_margin"][0, 0]), \
            (top_p, c, out["cut_margin"])


def check_exact_filtered(V=6, K=2, T=0.8, seed=19):
    """Exactness with top-k / top-p: with x_i drawn from the filtered draft
    distribution, the emitted token at every position follows the filtered
    target distribution (numpy filter) to 1e-12; dense and one-hot drafts,
    on logits with ties."""
    rng = np.random.default_rng(seed)
    l = (np.round(rng.standard_normal((K + 1, V)) * 3) / 2).astype(np.float32)
    d = (l[:K] + np.round(rng.standard_normal((K, V)) * 2) / 2).astype(np.float32)
    for top_k, top_p in ((4, 1.0), (0, 0.7), (5, 0.8)):
        p = np.array([np_filter(l[i], T, top_k, top_p) for i in range(K + 1)])
        q = np.array([np_filter(d[i], T, top_k, top_p) for i in range(K)])
        req = _Request(l, d, T, top_k=top_k, top_p=top_p)
        prefix = [int(np.argmax(p[j] * q[j])) for j in range(K)]
        for i in range(K + 1):
            emitted = np.zeros(V)
            for x in (range(V) if i < K else [0]):
                if i < K and q[i, x] == 0:
                    continue
                drafts = prefix[:i] + [x] + prefix[i + 1:] if i < K else list(prefix)
                theta, law = _emission_law(req, drafts, i)
                if i < K:
                    emitted[x] += q[i, x] * theta
                    emitted += q[i, x] * (1.0 - theta) * law
                else:
                    emitted = law
            np.testing.assert_allclose(emitted, p[i], rtol=0, atol=1e-12,
                                       err_msg="dense k=%d p=%g position %d" % (top_k, top_p, i))
        req = _Request(l, None, T, top_k=top_k, top_p=top_p)
        prefix = [int(np.argmax(p[j])) for j in range(K)]
        for i in range(K):
            for x in range(V):
                drafts = prefix[:i] + [x] + prefix[i + 1:]
                theta, law = _emission_law(req, drafts, i)
                assert abs(theta - min(1.0, p[i, x])) < 1e-12
                emitted = (1.0 - theta) * law
                emitted[x] += theta
                np.testing.assert_allclose(emitted, p[i], rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# typical acceptance
# ---------------------------------------------------------------------------

def check_golden_typical():
    g = _golden("typical_v5.json")
    rows = np.asarray(g["rows"])
    with np.errstate(divide="ignore"):
        lg = np.log(rows).astype(np.float32)
    chain = lg[:3][None]
    for case in g["chain"]:
        out = oracle.typical(chain, [case["draft_tokens"]], [case["uniforms"]], g["T"],
                             case["eps"], case["delta"])
        assert out["status"][0] == 0, out
        assert int(out["flags"][0][0]) == case.get("flag0", 0) and (out["flags"][0][1:] == 0).all()
        assert list(out["tokens"][0]) == case["tokens"], (case, out["tokens"][0])
        assert out["accept_len"][0] == case["accept_len"]
        np.testing.assert_allclose(out["accept_prob"][0], case["accept_prob"], atol=1e-6)
    tree_rows = lg[[0, 1, 2, 3]][None]
    for case in g["tree"]:
        out = oracle.tree_typical(tree_rows, g["tree_parent"], [case["node_tokens"]], [case["u"]],
                                  g["T"], case["eps"], case["delta"], 2)
        assert out["status"][0] == 0 and out["flags"][0] == 0, out
        assert list(out["tokens"][0]) == case["tokens"], (case, out["tokens"][0])
        assert list(out["path"][0]) == case["path"] and out["accept_len"][0] == case["accept_len"]


def check_typical_matches_scipy(seed=20):
    """Random rows: every tested position reports p(x), the decision is
    p(x) > min(eps, delta * exp(-H)) with H from scipy.stats.entropy, and the
    emitted token is the searchsorted draw from p_n."""
    import scipy.stats
    rng = np.random.default_rng(seed)
    B, K, V, T = 400, 4, 30, 0.8
    l = (rng.standard_normal((B, K + 1, V)) * 1.5).astype(np.float32)
    p = scipy.special.softmax(l.astype(np.float64) / T, axis=-1)
    am = np.argmax(l, axis=2)
    x = np.where(rng.random((B, K)) < 0.6, am[:, :K], rng.integers(0, V, (B, K))).astype(np.int32)
    u = rng.random((B, K + 1)).astype(np.float32)
    for eps, delta in ((0.09, 0.3), (0.3, 0.05), (0.02, 0.9)):
        out = oracle.typical(l, x, u, T, eps, delta)
        for b in range(B):
            n = int(out["accept_len"][b]) - 1
            for i in range(min(n + 1, K)):
                thr = min(eps, delta * np.exp(-scipy.stats.entropy(p[b, i])))
                px = p[b, i, x[b, i]]
                assert abs(out["accept_prob"][b, i] - px) < 1e-12
                if out["flags"][b, i] & oracle.FLAG_ACCEPT:
                    break
                assert (px > thr) == (i < n), (b, i, px, thr)
            if not (out["flags"][b] & oracle.FLAG_ACCEPT).any():
                assert out["tokens"][b, n] == _searchsorted_draw(p[b, n], float(u[b, K]))
                assert (out["tokens"][b, :n] == x[b, :n]).all()


def _typical_tree_brute(p, parent, node_tokens, u, eps, delta):
    """Enumerate root paths: a path counts when every node on it passes under
    its parent's distribution; the deepest, then the lowest end node."""
    import scipy.stats
    N = len(parent)
    thr = [min(eps, delta * np.exp(-scipy.stats.entropy(p[n]))) for n in range(N + 1)]
    best, best_d = 0, 0
    for end in range(1, N + 1):
        path, n = [], end
        while n:
            path.append(n)
            n = parent[n - 1]
        ok = all(p[parent[m - 1], node_tokens[m - 1]] > thr[parent[m - 1]] for m in path)
        if ok and len(path) > best_d:
            best, best_d = end, len(path)
    path, n = [], best
    while n:
        path.append(n)
        n = parent[n - 1]
    path = [0] + path[::-1]
    toks = [node_tokens[m - 1] for m in path[1:]] + [_searchsorted_draw(p[best], u)]
    return toks, path


def check_tree_typical_brute_force(seed=21):
    rng = np.random.default_rng(seed)
    for trial in range(40):
        N = int(rng.integers(1, 12))
        parent = [int(rng.integers(0, n)) for n in range(1, N + 1)]
        depth = [0] * (N + 1)
        for n in range(1, N + 1):
            depth[n] = depth[parent[n - 1]] + 1
        V, T = 6, 1.0
        l = (rng.standard_normal((1, N + 1, V)) * 1.2).astype(np.float32)
        p = scipy.special.softmax(l[0].astype(np.float64) / T, axis=-1)
        toks = rng.integers(0, V, size=(1, N)).astype(np.int32)
        u = float(rng.random())
        eps, delta = float(rng.choice([0.09, 0.2, 0.4])), float(rng.choice([0.3, 0.6, 1.0]))
        out = oracle.tree_typical(l, parent, toks, [u], T, eps, delta, max(depth))
        if out["flags"][0]:
            continue
        want_toks, want_path = _typical_tree_brute(p, parent, list(toks[0]), u, eps, delta)
        L = len(want_path)
        assert out["accept_len"][0] == L, (trial, out, want_path)
        assert list(out["path"][0, :L]) == want_path and list(out["tokens"][0, :L]) == want_toks


# ---------------------------------------------------------------------------
# n-gram proposer
# ---------------------------------------------------------------------------

def check_golden_ngram():
    g = _golden("ngram_small.json")
    for case in g["cases"]:
        ctx = case["context"]
        L = max(1, len(ctx) + 3)
        t = np.full((1, L), 99, np.int32)  # junk past the context is never read
        t[0, :len(ctx)] = ctx
        out = oracle.ngram(t, [len(ctx)], case["n_min"], case["n_max"], case["K"])
        k = len(case["drafts"])
        assert out["draft_lens"][0] == k, (case, out)
        assert list(out["drafts"][0, :k]) == case["drafts"] and (out["drafts"][0, k:] == -1).all()
        assert out["match"][0] == case["match"] and out["ngram"][0] == case["ngram"], (case, out)


def _ngram_numpy(c, n_min, n_max, K):
    """The same rule through numpy's sliding windows: starts s with
    s + n < len are the windows of c[:len-1]."""
    c = np.asarray(c)
    for n in range(n_max, n_min - 1, -1):
        if len(c) < n + 1:
            continue
        win = np.lib.stride_tricks.sliding_window_view(c[:-1], n)
        hit = np.flatnonzero((win == c[len(c) - n:]).all(axis=1))
        if hit.size:
            s = int(hit[0])
            return list(c[s + n:s + n + K]), s, n
    return [], -1, 0


def check_ngram_matches_numpy(seed=17):
    """Random contexts over small alphabets (many repeats): the oracle agrees
    with the sliding-window search, the drafts continue a real earlier
    occurrence, and no longer n-gram (up to n_max) occurs earlier."""
    rng = np.random.default_rng(seed)
    B, L = 300, 60
    for n_min, n_max, K in ((1, 4, 5), (2, 3, 2), (1, 1, 7), (3, 6, 4)):
        alpha = rng.integers(2, 6, size=B)
        t = (rng.integers(0, 1 << 30, size=(B, L)) % alpha[:, None]).astype(np.int32)
        lens = rng.integers(0, L + 1, size=B).astype(np.int32)
        out = oracle.ngram(t, lens, n_min, n_max, K)
        assert (out["status"] == 0).all()
        for b in range(B):
            c = t[b, :lens[b]]
            d, s, n = _ngram_numpy(c, n_min, n_max, K)
            k = int(out["draft_lens"][b])
            assert list(out["drafts"][b, :k]) == d and int(out["match"][b]) == s, (b, n_min, n_max)
            assert int(out["ngram"][b]) == n
            if s >= 0:
                assert (c[s:s + n] == c[len(c) - n:]).all() and s + n < len(c)
                assert k == min(K, len(c) - s - n) and k >= 1
    # a context length outside [0, L] is a per-request error
    out = oracle.ngram(np.zeros((3, 4), np.int32), [2, 5, -1], 1, 2, 3)
    assert list(out["status"]) == [0, oracle.BAD_DRAFT_LEN, oracle.BAD_DRAFT_LEN]
    assert list(out["draft_lens"]) == [1, 0, 0]


# ---------------------------------------------------------------------------
# tree
# ---------------------------------------------------------------------------

def _random_tree(rng, N):
    parent = []
    for n in range(1, N + 1):
        parent.append(int(rng.integers(0, n)))
    return np.asarray(parent, np.int32)


def _brute_force_tree(logits, parent, node_tokens):
    """Longest root path whose every node token equals the argmax of its
    parent's row (numpy argmax), by enumerating all root paths."""
    N = len(parent)
    best = [0]
    for n in range(1, N + 1):
        path = [n]
        while path[-1] != 0:
            path.append(int(parent[path[-1] - 1]))
        path = path[::-1]
        ok = all(node_tokens[c - 1] == int(np.argmax(logits[p])) for p, c in zip(path, path[1:]))
        if ok and len(path) > len(best):
            best = path
    toks = [int(np.argmax(logits[v])) for v in best]
    return best, toks


def check_tree_brute_force(seed=14):
    rng = np.random.default_rng(seed)
    for trial in range(60):
        N = int(rng.integers(1, 25))
        V = int(rng.integers(2, 9))
        parent = _random_tree(rng, N)
        depth = [0]
        for p in parent:
            depth.append(depth[p] + 1)
        D = max(depth)
        B = 6
        logits = rng.integers(0, 3, size=(B, N + 1, V)).astype(np.float32)
        tokens = np.zeros((B, N), np.int32)
        for b in range(B):
            for p in range(N + 1):
                ch = [c for c in range(1, N + 1) if parent[c - 1] == p]
                if not ch:
                    continue
                cand = [int(t) for t in rng.permutation(V)]
                if rng.random() < 0.8:  # make the matching child likely
                    a = int(np.argmax(logits[b, p]))
                    cand.remove(a)
                    cand.insert(int(rng.integers(0, min(len(ch), V))), a)
                while len(cand) < len(ch):  # more children than tokens: repeats
                    cand.append(int(rng.integers(0, V)))
                for c, t in zip(ch, cand):
                    tokens[b, c - 1] = t
        out = oracle.tree(logits, parent, tokens, D)
        for b in range(B):
            sib_distinct = all(len({int(tokens[b, c - 1]) for c in range(1, N + 1)
                                    if parent[c - 1] == p}) ==
                               sum(1 for c in range(1, N + 1) if parent[c - 1] == p)
                               for p in range(N + 1))
            if not sib_distinct:
                continue
            path, toks = _brute_force_tree(logits[b], parent, tokens[b])
            L = int(out["accept_len"][b])
            assert L == len(path), (trial, b, L, path)
            assert list(out["path"][b, :L]) == path
            assert list(out["tokens"][b, :L]) == toks
            assert (out["tokens"][b, L:] == -1).all() and (out["path"][b, L:] == -1).all()


def check_tree_errors():
    """Bad tokens and parent arrays that are not trees (a parent that is not
    an earlier node, or deeper than max_depth) are per-request statuses, in
    the greedy, typical and sampling tree walks alike; the other requests of
    the call are unaffected."""
    parent = np.array([0, 0, 1], np.int32)
    l = np.zeros((2, 4, 3), np.float32)
    toks = np.array([[0, 1, 2], [0, 3, 2]], np.int32)
    u = np.full((2, 4), 0.5)
    walks = [
        lambda par, D: oracle.tree(l, par, toks, D),
        lambda par, D: oracle.tree_typical(l, par, toks, u[:, 0], 1.0, 0.09, 0.3, D),
        lambda par, D: oracle.tree_sample(l, par, toks, u, 1.0, D),
    ]
    for walk in walks:
        out = walk(parent, 2)
        assert list(out["status"]) == [0, oracle.BAD_TOKEN]
        for bad in (np.array([0, 2, 1], np.int32), np.array([1, 0, 1], np.int32),
                    np.array([0, 0, -1], np.int32)):
            out = walk(bad, 2)
            assert out["status"][0] == oracle.BAD_TREE, bad
            assert out["accept_len"][0] == 0 and (out["tokens"][0] == -1).all()
        out = walk(parent, 1)  # depth 2 > max_depth 1
        assert out["status"][0] == oracle.BAD_TREE
        # one tree per request: request 0 valid, request 1 not a tree
        per = np.stack([parent, np.array([0, 3, 1], np.int32)])
        out = walk(per, 2)
        assert out["status"][0] == 0 and out["status"][1] == oracle.BAD_TREE


def check_per_request_trees(seed=23):
    """A [B, N] parent array (one tree per request) gives each request the
    result of a call with its own tree alone, for all three tree walks."""
    rng = np.random.default_rng(seed)
    B, N, V = 6, 9, 7
    parents = np.stack([_random_tree(rng, N) for _ in range(B)])
    D = N
    l = (rng.standard_normal((B, N + 1, V)) * 1.3).astype(np.float32)
    toks = rng.integers(0, V, size=(B, N)).astype(np.int32)
    for b in range(B):  # make some greedy walks go deep
        for n in range(1, N + 1):
            if rng.random() < 0.6:
                toks[b, n - 1] = int(np.argmax(l[b, parents[b, n - 1]]))
    u = rng.random((B, N + 1))
    both = [(lambda par, sl: oracle.tree(l[sl], par, toks[sl], D)),
            (lambda par, sl: oracle.tree_typical(l[sl], par, toks[sl], u[sl, 0], 1.0, 0.1, 0.4, D)),
            (lambda par, sl: oracle.tree_sample(l[sl], par, toks[sl], u[sl], 0.9, D))]
    for walk in both:
        full = walk(parents, slice(0, B))
        for b in range(B):
            one = walk(parents[b], slice(b, b + 1))
            for k in ("tokens", "path", "accept_len", "status"):
                assert (np.asarray(full[k][b]) == np.asarray(one[k][0])).all(), (b, k)


# ---------------------------------------------------------------------------
# lossless tree verification by rejection sampling
# ---------------------------------------------------------------------------

def _log_rows(rows):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(rows, np.float64)).astype(np.float32)


def check_golden_tree_sample():
    g = _golden("tree_sample_v4.json")
    l = _log_rows(g["rows"])[None]
    toks = np.asarray([g["node_tokens"]], np.int32)
    for case in g["cases"]:
        out = oracle.tree_sample(l, g["parent"], toks, np.asarray([case["uniforms"]]), g["T"],
                                 g["max_depth"])
        assert out["status"][0] == 0
        assert list(out["tokens"][0]) == case["tokens"], (case, out["tokens"][0])
        assert list(out["path"][0]) == case["path"], (case, out["path"][0])
        assert out["accept_len"][0] == case["accept_len"]
        np.testing.assert_allclose(out["accept_prob"][0], case["accept_prob"], atol=1e-6)


class _TreeRequest:
    """One tree request evaluated by the oracle for chosen uniforms."""

    def __init__(self, logits, parent, node_tokens, T):
        self.l = np.ascontiguousarray(logits[None], np.float32)
        self.parent = np.asarray(parent, np.int32)
        self.toks = np.asarray([node_tokens], np.int32)
        self.N = len(parent)
        self.T = T
        depth = [0]
        for pa in parent:
            depth.append(depth[pa] + 1)
        self.depth = depth

    def run(self, u):
        out = oracle.tree_sample(self.l, self.parent, self.toks, np.asarray([u]), self.T,
                                 max(self.depth))
        assert out["status"][0] == 0
        return out["path"][0], out["tokens"][0]


def _tree_emission_law(req, v):
    """Exact law of the token emitted after node v, the walk having reached
    v (uniform 0 for the tests on v's root path, the earlier siblings on that
    path rejected), by bisection over the uniforms of v's children in id
    order and then over the final draw's uniform.  None if v cannot be
    reached that way."""
    N, V = req.N, req.l.shape[2]
    chain, n = [], v
    while n:
        chain.append(n)
        n = int(req.parent[n - 1])
    u = [0.5] * (N + 1)
    for n in chain:  # accept the path, reject the earlier siblings
        u[n] = 0.0
        for c in range(1, n):
            if req.parent[c - 1] == req.parent[n - 1]:
                u[c] = _ONE_MINUS
    d = req.depth[v]
    path, _ = req.run(u)
    if path[d] != v:
        return None
    law, reach = np.zeros(V), 1.0
    children = [c for c in range(1, N + 1) if req.parent[c - 1] == v]
    for c in children:
        u[c] = 0.5

        def accepted(a, c=c):
            uu = list(u)
            uu[c] = a
            pth, _ = req.run(uu)
            return d + 1 < len(pth) and pth[d + 1] == c

        theta = _bisect(accepted)
        law[req.toks[0, c - 1]] += reach * theta
        reach *= 1.0 - theta
        u[c] = _ONE_MINUS
        if theta >= 1.0 or reach == 0.0:
            return law

    def token(s):
        uu = list(u)
        uu[0] = s
        pth, tk = req.run(uu)
        assert len(pth) <= d + 1 or pth[d + 1] < 0, "a rejected child was accepted"
        return int(tk[d])

    prev = 0.0
    for t in range(V):
        edge = 1.0 if t == V - 1 else _bisect(lambda s: token(s) <= t)
        law[t] += reach * (edge - prev)
        prev = edge
    return law


def check_exact_tree_sample(seed=24):
    """Exactness over a candidate tree: whatever node the walk stands on, the
    token emitted after it is distributed as that node's tempered target
    distribution, to 1e-12 - with repeated sibling tokens, tokens of zero
    probability, leaves and a node with a child for every token."""
    rng = np.random.default_rng(seed)
    cases = []
    for trial in range(4):
        N = int(rng.integers(3, 8))
        parent = list(_random_tree(rng, N))
        cases.append((parent, int(rng.integers(3, 6))))
    cases.append(([0, 0, 0, 0, 1, 1], 4))  # the root has a child for every token
    for ci, (parent, V) in enumerate(cases):
        N = len(parent)
        T = float(rng.choice([0.7, 1.0, 1.6]))
        l = (rng.standard_normal((N + 1, V)) * 1.2).astype(np.float32)
        toks = rng.integers(0, V, size=N).astype(np.int32)
        if ci == 4:
            toks[:4] = [2, 0, 3, 1]
        if ci == 1:
            toks[-1] = toks[0] if parent[-1] == parent[0] else toks[-1]
            l[0, 1] = -np.inf  # a zero-probability token at the root
        req = _TreeRequest(l, parent, toks, T)
        p = scipy.special.softmax(l.astype(np.float64) / T, axis=-1)
        checked = 0
        for v in range(N + 1):
            law = _tree_emission_law(req, v)
            if law is None:
                continue
            checked += 1
            np.testing.assert_allclose(law, p[v], rtol=0, atol=1e-12,
                                       err_msg="tree %s node %d" % (parent, v))
        assert checked >= 2, (parent, checked)


def check_tree_sample_chain_is_onehot_verify(seed=25):
    """A chain-shaped tree (node n's parent is n-1) is one-hot rejection
    sampling over K = N positions: the same tokens and acceptance
    probabilities as the chain verification with the uniforms remapped
    (node n's test uses chain column n-1, the final draw column K)."""
    rng = np.random.default_rng(seed)
    B, N, V, T = 200, 4, 50, 0.8
    l = (rng.standard_normal((B, N + 1, V)) * 2.0).astype(np.float32)
    x = np.where(rng.random((B, N)) < 0.5, np.argmax(l[:, :N], axis=2),
                 rng.integers(0, V, size=(B, N))).astype(np.int32)
    u = rng.random((B, N + 1))
    chain = oracle.sample(l, None, x, np.concatenate([u[:, 1:], u[:, :1]], axis=1), T)
    tree = oracle.tree_sample(l, np.arange(N, dtype=np.int32), x, u, T, N)
    assert (tree["tokens"] == chain["tokens"]).all()
    assert (tree["accept_len"] == chain["accept_len"]).all()
    for b in range(B):
        L = int(chain["accept_len"][b])
        tested = min(L, N)
        np.testing.assert_allclose(tree["accept_prob"][b, 1:tested + 1],
                                   chain["accept_prob"][b, :tested], rtol=0, atol=1e-14)
        assert list(tree["path"][b, :L]) == list(range(L))


def check_flips_invert_tests(seed=26):
    """The checking hook: flipping a test the request reaches inverts its
    outcome (and nothing before it); flipping a test it never reaches
    changes nothing.  Chains (rejection sampling and typical acceptance) and
    trees (sampling and typical acceptance)."""
    rng = np.random.default_rng(seed)
    B, K, V, T = 64, 3, 30, 1.0
    l = (rng.standard_normal((B, K + 1, V)) * 1.5).astype(np.float32)
    d = (l[:, :K] + rng.standard_normal((B, K, V)) * 0.6).astype(np.float32)
    x = np.argmax(d, axis=2).astype(np.int32)
    u = rng.random((B, K + 1))
    for run in (lambda f: oracle.sample(l, d, x, u, T, flip=f),
                lambda f: oracle.sample(l, None, x, u, T, flip=f),
                lambda f: oracle.typical(l, x, u, T, 0.09, 0.3, flip=f)):
        base = run(None)
        for i in range(K):
            f = np.zeros((B, K), np.uint8)
            f[:, i] = 1
            out = run(f)
            for b in range(B):
                L0, L1 = int(base["accept_len"][b]), int(out["accept_len"][b])
                if L0 < i + 1:  # test i not reached
                    assert (out["tokens"][b] == base["tokens"][b]).all()
                elif L0 > i + 1:  # accepted at i: now rejected there
                    assert L1 == i + 1 and (out["tokens"][b, :i] == base["tokens"][b, :i]).all()
                else:  # rejected at i: now accepted there
                    assert L1 > i + 1 and (out["tokens"][b, :i + 1] == x[b, :i + 1]).all()
    parent = np.array([0, 0, 1, 1, 2, 3], np.int32)
    N = parent.size
    lt = (rng.standard_normal((B, N + 1, V)) * 1.5).astype(np.float32)
    toks = np.argsort(-lt[:, parent], axis=2)[:, np.arange(N), np.array([0, 1, 0, 1, 0, 0])]
    toks = np.ascontiguousarray(toks, dtype=np.int32)
    ut = rng.random((B, N + 1))
    # trees: a flipped node on the walked path leaves it; for the sampling
    # walk, a tested node off the path joins it and an untested one changes
    # nothing
    for run, sampling in ((lambda f: oracle.tree_sample(lt, parent, toks, ut, T, 3, flip=f), True),
                          (lambda f: oracle.tree_typical(lt, parent, toks, ut[:, 0], T, 0.09, 0.3,
                                                         3, flip=f), False)):
        base = run(None)
        moved = 0
        for n in range(1, N + 1):
            f = np.zeros((B, N + 1), np.uint8)
            f[:, n] = 1
            out = run(f)
            for b in range(B):
                on_path = n in list(base["path"][b])
                if on_path:
                    assert n not in list(out["path"][b]), (b, n)
                    moved += 1
                elif sampling and base["accept_prob"][b, n] >= 0:
                    assert n in list(out["path"][b]), (b, n)
                    moved += 1
                elif sampling:
                    assert (out["tokens"][b] == base["tokens"][b]).all()
        assert moved > B, moved


def check_probes(seed=28):
    """The probe that checks a draw made elsewhere: for the emitted token the
    reported CDF step contains the draw's uniform; for any token it is the
    step of the draw's weights computed with numpy (one-hot residual p_n
    without x_n, or the bonus p_K; typical acceptance: p_n; the tree
    sampler: the residual at the final node)."""
    rng = np.random.default_rng(seed)
    B, K, V, T = 80, 2, 30, 1.1
    l = (rng.standard_normal((B, K + 1, V)) * 1.5).astype(np.float32)
    x = np.where(rng.random((B, K)) < 0.5, np.argmax(l[:, :K], axis=2),
                 rng.integers(0, V, size=(B, K))).astype(np.int32)
    u = rng.random((B, K + 1))
    p = scipy.special.softmax(l.astype(np.float64) / T, axis=-1)

    def step(w, t):
        c = np.concatenate([[0.0], np.cumsum(w)]) / w.sum()
        return c[t], c[t + 1]

    for kind in ("sample", "typical"):
        run = (lambda pt: oracle.sample(l, None, x, u, T, probe_tokens=pt)) if kind == "sample" \
            else (lambda pt: oracle.typical(l, x, u, T, 0.09, 0.3, probe_tokens=pt))
        base = run(None)
        n = base["accept_len"] - 1
        own = run(base["tokens"][np.arange(B), n])["probe"]
        assert ((own[:, 0] <= u[:, K]) & (u[:, K] < own[:, 1])).all(), kind
        other = rng.integers(0, V, size=B).astype(np.int32)
        pr = run(other)["probe"]
        for b in range(B):
            w = p[b, n[b]].copy()
            if kind == "sample" and n[b] < K:
                w[x[b, n[b]]] = 0.0
            lo, hi = step(w, other[b])
            assert abs(pr[b, 0] - lo) < 1e-12 and abs(pr[b, 1] - hi) < 1e-12, (kind, b)
    parent = np.array([0, 0, 1], np.int32)
    lt = (rng.standard_normal((B, 4, V)) * 1.5).astype(np.float32)
    toks = np.ascontiguousarray(np.argsort(-lt[:, parent], axis=2)[:, np.arange(3), [0, 1, 0]],
                                dtype=np.int32)
    ut = rng.random((B, 4))
    base = oracle.tree_sample(lt, parent, toks, ut, T, 2)
    L = base["accept_len"]
    own = oracle.tree_sample(lt, parent, toks, ut, T, 2,
                             probe_tokens=base["tokens"][np.arange(B), L - 1])["probe"]
    assert ((own[:, 0] <= ut[:, 0]) & (ut[:, 0] < own[:, 1])).all()


ALL_CHECKS = [
    check_softmax_matches_scipy, check_argmax_matches_numpy,
    check_inverse_cdf_matches_searchsorted, check_golden_sampling, check_golden_greedy,
    check_golden_tree, check_golden_compact, check_exact_dense, check_exact_onehot,
    check_invariants, check_onehot_accept_iff_u_below_p,
    check_zero_probability_draft_rejected, check_temperature_to_zero_is_greedy,
    check_errors, check_tree_brute_force, check_tree_errors, check_golden_masked,
    check_mask_layout, check_exact_masked, check_golden_ngram, check_ngram_matches_numpy,
    check_golden_topk_topp, check_filter_matches_numpy, check_exact_filtered,
    check_golden_typical, check_typical_matches_scipy, check_tree_typical_brute_force,
    check_per_request_trees, check_golden_tree_sample, check_exact_tree_sample,
    check_tree_sample_chain_is_onehot_verify, check_flips_invert_tests, check_forced_cut,
    check_probes,
]
