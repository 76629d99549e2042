"""Comparing the CUDA path with the fp64 oracle.

The fp32 GPU arithmetic and the fp64 oracle can only disagree where a
uniform falls within rounding distance of a decision boundary.  The oracle
flags those places (a test whose uniform lies within 1e-5 * theta of its
threshold theta; a draw whose u * W lies within 1e-5 * W of an edge of the
chosen token's CDF step; a top-p cut whose mass in front lies within 1e-5 of
top_p), and the comparison verifies the GPU's result there instead of
excluding it:

  * statuses equal; a request with a data error emits nothing on both sides;
  * acceptance tests: where the GPU decided a test differently, that test
    must be one the oracle flags; the oracle is then run again with that
    test's outcome flipped (and so on for later flagged tests the new branch
    reaches), and the GPU must match that run exactly.  A test decided
    differently that the oracle does not flag is an error;
  * top-k / top-p cuts: the GPU reports each row's cut value; the oracle
    runs with those cuts forced and reports each one's distance from the
    rule (0 for the rule's own cut).  A cut that is not admissible, or that
    differs from the rule's by more than STRICT_TOL of mass, is an error;
  * draws: the token must equal the oracle's; where it does not, the
    oracle's draw must be flagged with a margin of at most STRICT_TOL, and
    the GPU's token's exact (fp64) CDF step, from the oracle's probe, must
    come within FLAG_TOL * W of u * W; the differing draws are counted by
    margin band, and in a flag-rate run they may be at most MAX_DIFFER_RATE
    of the positions;
  * accept probabilities within PROB_ATOL, at every position (-1 where a
    position was not tested).
Greedy and tree-greedy verification are compared bit-exactly.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import oracle

PROB_ATOL = 1e-5
FLAG_TOL = 1e-5     # the oracle's flag band
STRICT_TOL = 1e-6   # a GPU result may leave the oracle's only within this margin
BANDS = (1e-5, 1e-6, 1e-7, 1e-8)
# Draws that differ from the oracle's (each within STRICT_TOL and verified)
# may be at most this share of the positions in a flag-rate run: the oracle
# alone puts 7.8e-3 of the draws of the 152064-token one-hot workload within
# 1e-6 of a step edge, where an fp32 sampler may legitimately land on either
# side; the GPU has differed on at most 4.1e-4.
MAX_DIFFER_RATE = 1e-3
MIN_RATE_POSITIONS = 10000  # the rate is asserted over runs at least this large


def to_device(wl, device="cuda"):
    """Torch CUDA tensors of a synth.Workload (bf16 from the raw bit patterns)."""
    def logits(a):
        if a is None:
            return None
        if wl.dtype == "bf16":
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(a).to(device)

    d = dict(target=logits(wl.target), draft=logits(wl.draft))
    for name in ("draft_tokens", "draft_lens", "uniforms", "node_tokens"):
        v = getattr(wl, name)
        d[name] = None if v is None else torch.from_numpy(np.ascontiguousarray(v)).to(device)
    d["token_mask"] = None if wl.token_mask is None else torch.from_numpy(
        np.ascontiguousarray(wl.token_mask).view(np.int32)).to(device)
    if getattr(wl, "parent", None) is not None:
        d["parent"] = torch.from_numpy(np.ascontiguousarray(wl.parent, dtype=np.int32)).to(device)
    return d


@dataclass
class SampleReport:
    requests: int = 0
    positions: int = 0
    acc_flagged: int = 0      # acceptance tests within 1e-5 of theta
    acc_flipped: int = 0      # ... that the GPU decided the other way (verified)
    cut_differ: int = 0       # top-p cuts the GPU placed one class off (verified)
    cdf_flagged: int = 0      # final draws within 1e-5 * W of a CDF edge
    cdf_differ: int = 0       # ... whose GPU token differs from the oracle's (verified)
    differ_bands: list = field(default_factory=lambda: [0] * (len(BANDS) + 1))
    errors: list = field(default_factory=list)

    def band(self, margin):
        """Count a differing draw by the oracle's margin: (1e-6, 1e-5],
        (1e-7, 1e-6], (1e-8, 1e-7], <= 1e-8 (and > 1e-5, never allowed)."""
        for k, edge in enumerate(BANDS[1:]):
            if margin > edge:
                self.differ_bands[k] += 1
                return
        self.differ_bands[len(BANDS) - 1] += 1

    def merge(self, o):
        for k in ("requests", "positions", "acc_flagged", "acc_flipped", "cut_differ",
                  "cdf_flagged", "cdf_differ"):
            setattr(self, k, getattr(self, k) + getattr(o, k))
        self.differ_bands = [a + b for a, b in zip(self.differ_bands, o.differ_bands)]
        self.errors += o.errors

    def summary(self):
        bands = ", ".join("%s: %d" % (lbl, n) for lbl, n in zip(
            ("(1e-6,1e-5]", "(1e-7,1e-6]", "(1e-8,1e-7]", "<=1e-8"), self.differ_bands))
        return ("%d requests, %d positions: %d acceptance tests flagged (%d taken the other way, "
                "verified), %d top-p cuts one class off (verified), %d draws CDF-flagged of which "
                "%d differ from the oracle (verified; by oracle margin %s)"
                % (self.requests, self.positions, self.acc_flagged, self.acc_flipped,
                   self.cut_differ, self.cdf_flagged, self.cdf_differ, bands))


def _sub(a, idx):
    return None if a is None else np.ascontiguousarray(a[idx])


def _run_sample(wl, idx, T, threads, flips=None, cuts=None, probes=None):
    return oracle.sample(_sub(wl.target, idx), _sub(wl.draft, idx), _sub(wl.draft_tokens, idx),
                         _sub(wl.uniforms, idx), T, draft_lens=_sub(wl.draft_lens, idx),
                         token_mask=_sub(wl.token_mask, idx), top_k=wl.top_k,
                         top_p=float(np.float32(wl.top_p)), flip=flips, cut_logits=cuts,
                         probe_tokens=probes, threads=threads)


def _window_ok(lo, hi, u):
    return (hi > lo) & (lo <= u + FLAG_TOL) & (hi >= u - FLAG_TOL)


def compare_sample(wl, gpu, temperature=None, threads=16) -> SampleReport:
    """Rejection-sampling (or, at temperature 0, greedy) results of the GPU
    against the oracle on the same inputs (the module docstring's rule)."""
    T = wl.T if temperature is None else temperature
    K, V = wl.K, wl.V
    g_tok = gpu.tokens.cpu().numpy()
    g_len = gpu.accept_len.cpu().numpy()
    g_st = gpu.status.cpu().numpy() if gpu.status is not None else None
    g_prob = gpu.accept_prob.cpu().numpy() if gpu.accept_prob is not None else None
    cuts = None
    if getattr(gpu, "cut", None) is not None:
        cuts = gpu.cut.cpu().numpy().astype(np.float64)
    B = g_tok.shape[0]
    rep = SampleReport(requests=B, positions=B * (K + 1))
    everyone = np.arange(B)
    ref = _run_sample(wl, everyone, T, threads, cuts=cuts)
    if T == 0:
        for b in range(B):
            if g_st is not None and g_st[b] != ref["status"][b]:
                rep.errors.append((b, "status %d vs oracle %d" % (g_st[b], ref["status"][b])))
            elif g_len[b] != ref["accept_len"][b] or not (g_tok[b] == ref["tokens"][b]).all():
                rep.errors.append((b, "greedy %s vs oracle %s"
                                   % (g_tok[b].tolist(), ref["tokens"][b].tolist())))
        return rep
    rep.acc_flagged = int(((ref["flags"] & oracle.FLAG_ACCEPT) != 0).sum())
    flips = np.zeros((B, K), np.uint8)
    bad = np.zeros(B, bool)
    active = []
    for b in range(B):
        st = int(ref["status"][b])
        if g_st is not None and int(g_st[b]) != st:
            rep.errors.append((b, "status %d vs oracle %d" % (g_st[b], st)))
            bad[b] = True
        elif st:
            if g_len[b] != 0 or (g_tok[b] != -1).any():
                rep.errors.append((b, "a request with a data error emitted tokens"))
            bad[b] = True
        else:
            active.append(b)
    # follow the GPU's branch through flagged tests
    for _ in range(K + 1):
        redo = []
        for b in active:
            if bad[b]:
                continue
            Lr, Lg = int(ref["accept_len"][b]), int(g_len[b])
            if Lr == Lg:
                continue
            j = min(Lr, Lg) - 1  # both reached test j and decided it differently
            if j < 0 or j >= K or flips[b, j] or not ref["flags"][b, j] & oracle.FLAG_ACCEPT:
                rep.errors.append((b, "accept_len %d vs oracle %d at an unflagged test"
                                   % (Lg, Lr)))
                bad[b] = True
                continue
            flips[b, j] = 1
            redo.append(b)
        if not redo:
            break
        idx = np.asarray(redo)
        alt = _run_sample(wl, idx, T, threads, flips=flips[idx],
                          cuts=None if cuts is None else cuts[idx])
        for k, v in alt.items():
            ref[k][idx] = v
    # compare what must match, and collect the differing draws
    probe_idx, probe_tok = [], []
    for b in active:
        if bad[b]:
            continue
        L = int(g_len[b])
        n = L - 1
        rep.acc_flipped += int(flips[b].any())
        if L != int(ref["accept_len"][b]):
            rep.errors.append((b, "accept_len %d vs oracle %d" % (L, ref["accept_len"][b])))
            continue
        rt = ref["tokens"][b]
        same = g_tok[b] == rt
        cdf = bool(ref["flags"][b, n] & oracle.FLAG_CDF)
        rep.cdf_flagged += int(cdf)
        if not same[:n].all() or not same[n + 1:].all():
            rep.errors.append((b, "tokens %s vs oracle %s" % (g_tok[b].tolist(), rt.tolist())))
        elif not same[n]:
            margin = float(ref["margins"][b, K])
            if not cdf or margin > STRICT_TOL or not 0 <= g_tok[b, n] < V:
                rep.errors.append((b, "draw %d vs oracle %d at margin %.2e"
                                   % (g_tok[b, n], rt[n], margin)))
            else:
                rep.cdf_differ += 1
                rep.band(margin)
                probe_idx.append(b)
                probe_tok.append(int(g_tok[b, n]))
        if g_prob is not None:
            diff = np.abs(g_prob[b] - ref["accept_prob"][b])
            if not (diff <= PROB_ATOL).all():
                rep.errors.append((b, "accept_prob max diff %.3g" % diff.max()))
        if cuts is not None:
            cm = ref["cut_margin"][b]
            reached = cm != -1.0
            if np.isnan(cm[reached]).any():
                rep.errors.append((b, "a GPU cut the oracle cannot admit: %s" % cuts[b].tolist()))
            elif (cm[reached] > STRICT_TOL).any():
                rep.errors.append((b, "a GPU cut %.2e of mass off the rule" % cm[reached].max()))
            else:
                rep.cut_differ += int((cm[reached] > 0).sum())
    if probe_idx:  # the GPU's token's exact CDF step, in the branch the GPU took
        idx = np.asarray(probe_idx)
        out = _run_sample(wl, idx, T, threads, flips=flips[idx],
                          cuts=None if cuts is None else cuts[idx],
                          probes=np.asarray(probe_tok, np.int32))
        u = wl.uniforms[idx, K].astype(np.float64)
        ok = _window_ok(out["probe"][:, 0], out["probe"][:, 1], u)
        for j in np.nonzero(~ok)[0]:
            rep.errors.append((int(idx[j]), "GPU draw %d outside the window: step [%.9f, %.9f) "
                               "u %.9f" % (probe_tok[j], out["probe"][j, 0], out["probe"][j, 1],
                                           u[j])))
    return rep


def assert_report(rep: SampleReport, max_flag_rate=None):
    assert not rep.errors, "%d mismatching requests, first: %s" % (len(rep.errors), rep.errors[:5])
    if max_flag_rate is not None:
        assert rep.acc_flagged <= max_flag_rate * rep.positions, rep.summary()
        if rep.positions >= MIN_RATE_POSITIONS:
            assert rep.cdf_differ <= MAX_DIFFER_RATE * rep.positions, rep.summary()


def check_sample(wl, gpu, temperature=None, threads=16, flag_rate=None) -> SampleReport:
    rep = compare_sample(wl, gpu, temperature=temperature, threads=threads)
    assert_report(rep, flag_rate)
    return rep


# ---------------------------------------------------------------------------
# typical acceptance (chains)
# ---------------------------------------------------------------------------

def compare_typical(wl, gpu, eps, delta, threads=16) -> SampleReport:
    """Typical acceptance on chains: the same rule as compare_sample - a test
    decided differently must be flagged, and the GPU must match the oracle
    with it flipped; a differing draw must be flagged within STRICT_TOL and
    land in its exact CDF window; p(x) within PROB_ATOL."""
    K, V, T = wl.K, wl.V, wl.T
    g_tok, g_len = gpu.tokens.cpu().numpy(), gpu.accept_len.cpu().numpy()
    g_st, g_prob = gpu.status.cpu().numpy(), gpu.accept_prob.cpu().numpy()
    B = g_tok.shape[0]

    def run(idx, flips=None, probes=None):
        return oracle.typical(_sub(wl.target, idx), _sub(wl.draft_tokens, idx),
                              _sub(wl.uniforms, idx), T, eps, delta,
                              draft_lens=_sub(wl.draft_lens, idx), flip=flips,
                              probe_tokens=probes, threads=threads)

    rep = SampleReport(requests=B, positions=B * (K + 1))
    ref = run(np.arange(B))
    rep.acc_flagged = int(((ref["flags"] & oracle.FLAG_ACCEPT) != 0).sum())
    flips = np.zeros((B, K), np.uint8)
    bad = np.zeros(B, bool)
    for b in range(B):
        if g_st[b] != ref["status"][b]:
            rep.errors.append((b, "status"))
            bad[b] = True
        elif ref["status"][b]:
            bad[b] = True
    for _ in range(K + 1):
        redo = []
        for b in range(B):
            Lr, Lg = int(ref["accept_len"][b]), int(g_len[b])
            if bad[b] or Lr == Lg:
                continue
            j = min(Lr, Lg) - 1
            if j < 0 or j >= K or flips[b, j] or not ref["flags"][b, j] & oracle.FLAG_ACCEPT:
                rep.errors.append((b, "accept_len %d vs %d at an unflagged test" % (Lg, Lr)))
                bad[b] = True
                continue
            flips[b, j] = 1
            redo.append(b)
        if not redo:
            break
        idx = np.asarray(redo)
        alt = run(idx, flips[idx])
        for k, v in alt.items():
            ref[k][idx] = v
    probe_idx, probe_tok = [], []
    for b in range(B):
        if bad[b]:
            continue
        L = int(g_len[b])
        n = L - 1
        rep.acc_flipped += int(flips[b].any())
        same = g_tok[b] == ref["tokens"][b]
        cdf = bool(ref["flags"][b, n] & oracle.FLAG_CDF)
        rep.cdf_flagged += int(cdf)
        if L != ref["accept_len"][b] or not same[:n].all() or not same[n + 1:].all():
            rep.errors.append((b, "tokens %s vs %s" % (g_tok[b].tolist(),
                                                        ref["tokens"][b].tolist())))
            continue
        if not same[n]:
            margin = float(ref["margins"][b])
            if not cdf or margin > STRICT_TOL or not 0 <= g_tok[b, n] < V:
                rep.errors.append((b, "draw %d vs %d at margin %.2e"
                                   % (g_tok[b, n], ref["tokens"][b, n], margin)))
            else:
                rep.cdf_differ += 1
                rep.band(margin)
                probe_idx.append(b)
                probe_tok.append(int(g_tok[b, n]))
        diff = np.abs(g_prob[b] - ref["accept_prob"][b])
        if not (diff <= PROB_ATOL).all():
            rep.errors.append((b, "p(x) max diff %.3g" % diff.max()))
    if probe_idx:
        idx = np.asarray(probe_idx)
        out = run(idx, flips[idx], np.asarray(probe_tok, np.int32))
        ok = _window_ok(out["probe"][:, 0], out["probe"][:, 1],
                        wl.uniforms[idx, K].astype(np.float64))
        for j in np.nonzero(~ok)[0]:
            rep.errors.append((int(idx[j]), "GPU draw outside its window"))
    return rep


# ---------------------------------------------------------------------------
# trees
# ---------------------------------------------------------------------------

def _tree_compare(g, ref, b, u_draw, rep, V):
    """Path, tokens and length of tree request b against one oracle run;
    returns None on a match, "draw" when only a CDF-flagged draw differs (to
    be verified), else a message."""
    L = int(g["accept_len"][b])
    if L != int(ref["accept_len"][b]) or not (g["path"][b] == ref["path"][b]).all():
        return "path %s vs oracle %s" % (g["path"][b].tolist(), ref["path"][b].tolist())
    same = g["tokens"][b] == ref["tokens"][b]
    n = L - 1
    if not same[:n].all() or not same[n + 1:].all():
        return "tokens %s vs oracle %s" % (g["tokens"][b].tolist(), ref["tokens"][b].tolist())
    if same[n]:
        return None
    flagged = ref["flags"][b] & oracle.FLAG_CDF
    if not flagged or ref["margins"][b] > STRICT_TOL or not 0 <= g["tokens"][b, n] < V:
        return "draw %d vs oracle %d (margin %.2e)" % (g["tokens"][b, n], ref["tokens"][b, n],
                                                      ref["margins"][b])
    return "draw"


def compare_tree(wl, gpu, kind, T, eps=0.0, delta=0.0, threads=16, parent=None) -> SampleReport:
    """Tree verification by typical acceptance ("typical") or rejection
    sampling ("sample") against the oracle.  A node test decided differently
    must be one the oracle flags: the oracle is run again with it flipped
    (the sampling walk: the first test on the common path decided
    differently; typical acceptance: subsets of the flagged tests), and the
    GPU must match.  A differing draw must be CDF-flagged within STRICT_TOL
    and land in its exact window."""
    par = wl.parent if parent is None else parent
    g = {k: getattr(gpu, k).cpu().numpy() for k in ("tokens", "accept_len", "path", "status")}
    B, V = g["tokens"].shape[0], wl.V
    N = wl.node_tokens.shape[1]
    u = np.asarray(wl.uniforms)

    def run(idx, flips=None, probes=None):
        p = par if np.ndim(par) == 1 else np.ascontiguousarray(np.asarray(par)[idx])
        if kind == "sample":
            return oracle.tree_sample(_sub(wl.target, idx), p, _sub(wl.node_tokens, idx),
                                      _sub(u, idx), T, wl.max_depth, flip=flips,
                                      probe_tokens=probes, threads=threads)
        return oracle.tree_typical(_sub(wl.target, idx), p, _sub(wl.node_tokens, idx),
                                   _sub(u, idx), T, eps, delta, wl.max_depth, flip=flips,
                                   probe_tokens=probes, threads=threads)

    rep = SampleReport(requests=B, positions=B)
    ref = run(np.arange(B))
    rep.acc_flagged = int(((ref["node_flags"] & oracle.FLAG_ACCEPT) != 0).sum())
    flips = np.zeros((B, N + 1), np.uint8)
    probe_idx, probe_tok = [], []
    for b in range(B):
        if g["status"][b] != ref["status"][b]:
            rep.errors.append((b, "status %d vs oracle %d" % (g["status"][b], ref["status"][b])))
            continue
        if ref["status"][b]:
            if g["accept_len"][b] != 0 or (g["tokens"][b] != -1).any():
                rep.errors.append((b, "a request with a data error emitted tokens"))
            continue
        mine = {k: v[b:b + 1].copy() for k, v in ref.items()}
        fl = np.zeros((1, N + 1), np.uint8)
        gb = {k: v[b:b + 1] for k, v in g.items()}
        verdict = _tree_compare(gb, mine, 0, None, rep, V)
        if kind == "sample":
            for _ in range(N):  # the walk: flip the first test on the common path it decided
                if verdict in (None, "draw"):  # differently, if that test is flagged
                    break
                gp, rp = list(gb["path"][0]), list(mine["path"][0])
                d = 0
                while d < len(gp) and d < len(rp) and gp[d] == rp[d] and gp[d] >= 0:
                    d += 1
                cand = [x for x in (gp[d] if d < len(gp) else -1, rp[d] if d < len(rp) else -1)
                        if x > 0]
                node = min(cand) if cand else -1
                if node <= 0 or not mine["node_flags"][0, node] & oracle.FLAG_ACCEPT or fl[0, node]:
                    break
                fl[0, node] = 1
                mine = run(np.asarray([b]), fl)
                verdict = _tree_compare(gb, mine, 0, None, rep, V)
        else:  # typical acceptance: subsets of the flagged tests, breadth first
            queue, runs = [], 0
            for n in np.nonzero(mine["node_flags"][0] & oracle.FLAG_ACCEPT)[0]:
                queue.append(frozenset([int(n)]))
            while verdict not in (None, "draw") and queue and runs < 16:
                S = queue.pop(0)
                fl = np.zeros((1, N + 1), np.uint8)
                fl[0, sorted(S)] = 1
                mine = run(np.asarray([b]), fl)
                runs += 1
                verdict = _tree_compare(gb, mine, 0, None, rep, V)
                for n in np.nonzero(mine["node_flags"][0] & oracle.FLAG_ACCEPT)[0]:
                    if int(n) not in S and len(S) < 3:
                        queue.append(S | {int(n)})
        if verdict not in (None, "draw"):
            rep.errors.append((b, verdict))
            continue
        flips[b] = fl[0]
        rep.acc_flipped += int(fl.any())
        rep.cdf_flagged += int(bool(mine["flags"][0] & oracle.FLAG_CDF))
        if verdict == "draw":
            rep.cdf_differ += 1
            rep.band(float(mine["margins"][0]))
            L = int(g["accept_len"][b])
            probe_idx.append(b)
            probe_tok.append(int(g["tokens"][b, L - 1]))
    if probe_idx:
        idx = np.asarray(probe_idx)
        out = run(idx, flips[idx], np.asarray(probe_tok, np.int32))
        uu = (u[idx, 0] if kind == "sample" else u[idx]).astype(np.float64)
        ok = _window_ok(out["probe"][:, 0], out["probe"][:, 1], uu)
        for j in np.nonzero(~ok)[0]:
            rep.errors.append((int(idx[j]), "GPU draw outside its window"))
    return rep


def compare_compaction(gpu, K):
    tok = gpu.tokens.cpu().numpy()
    L = gpu.accept_len.cpu().numpy()
    cu, packed, bid = oracle.compact(tok, L)
    assert (gpu.cu_accept.cpu().numpy() == cu).all(), "cu_accept differs"
    assert (gpu.packed.cpu().numpy() == packed).all(), "packed tokens differ"
    assert (gpu.batch_id.cpu().numpy() == bid).all(), "batch ids differ"
