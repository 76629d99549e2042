"""Helpers for comparing the CUDA path with the fp64 oracle.

Comparison rule for rejection sampling (the fp32 GPU arithmetic and the
fp64 oracle can only disagree where a uniform falls within rounding distance
of a decision boundary):
  * statuses equal; a request with a data error emits nothing on both sides;
  * unflagged request: token row, accept_len and accept probabilities
    (|diff| <= 1e-5) equal;
  * the oracle flags an acceptance test at position i (u within 1e-5 * theta
    of theta): positions before i must match and the GPU must have reached
    position i; positions i.. are excluded;
  * the oracle flags the final draw at position n (u*W within 1e-5 * W of an
    edge of the chosen token's CDF step - which always holds when the draw
    lands on a token lighter than 1e-5 of the total): everything but token n
    must match, and token n is still checked: it must equal the oracle's
    token unless the oracle's margin is below STRICT_TOL, and in any case its
    exact (fp64) CDF step must lie within 1e-5 * W of u*W (verify_draws).
Greedy and tree verification are compared bit-exactly.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import oracle

PROB_ATOL = 1e-5
FLAG_TOL = 1e-5     # the oracle's flag band
STRICT_TOL = 1e-6   # flagged draws farther than this from an edge must still match


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
    return d


def oracle_sample(wl, threads=8, temperature=None):
    T = wl.T if temperature is None else temperature
    return oracle.sample(wl.target, wl.draft, wl.draft_tokens, wl.uniforms, T,
                         draft_lens=wl.draft_lens, threads=threads, token_mask=wl.token_mask,
                         top_k=wl.top_k, top_p=float(np.float32(wl.top_p)))


@dataclass
class SampleReport:
    requests: int = 0
    positions: int = 0
    acc_flagged: int = 0      # acceptance tests within 1e-5 of theta
    cut_flagged: int = 0      # top-p cuts within 1e-5 of moving
    excluded: int = 0         # positions not compared because of them
    cdf_flagged: int = 0      # final draws within 1e-5 * W of a CDF edge
    cdf_differ: int = 0       # ... whose GPU token differs from the oracle's
    errors: list = field(default_factory=list)
    to_verify: list = field(default_factory=list)  # (b, n, gpu token)

    @property
    def flagged(self):
        return self.acc_flagged + self.cdf_flagged

    def merge(self, o):
        for k in ("requests", "positions", "acc_flagged", "cut_flagged", "excluded", "cdf_flagged",
                  "cdf_differ"):
            setattr(self, k, getattr(self, k) + getattr(o, k))
        self.errors += o.errors

    def summary(self):
        return ("%d requests, %d positions: %d acceptance-flagged, %d top-p cuts flagged (%d "
                "positions excluded), %d draws CDF-flagged of which %d differ from the oracle "
                "(all verified)" % (self.requests, self.positions, self.acc_flagged,
                                    self.cut_flagged, self.excluded, self.cdf_flagged,
                                    self.cdf_differ))


def compare_sample(ref, gpu, K, V, greedy=False) -> SampleReport:
    g_tok = gpu.tokens.cpu().numpy()
    g_len = gpu.accept_len.cpu().numpy()
    g_st = gpu.status.cpu().numpy() if gpu.status is not None else None
    g_prob = gpu.accept_prob.cpu().numpy() if gpu.accept_prob is not None else None
    B = g_tok.shape[0]
    rep = SampleReport(requests=B, positions=B * (K + 1))
    for b in range(B):
        st = int(ref["status"][b])
        if g_st is not None and int(g_st[b]) != st:
            rep.errors.append((b, "status %d vs oracle %d" % (g_st[b], st)))
            continue
        if st:
            if g_len[b] != 0 or (g_tok[b] != -1).any():
                rep.errors.append((b, "error request emitted tokens"))
            continue
        L = int(ref["accept_len"][b])
        flags = ref["flags"][b]
        acc_flag = next((i for i in range(K + 1)
                         if flags[i] & (oracle.FLAG_ACCEPT | oracle.FLAG_CUT)), None)
        cut = acc_flag is not None and bool(flags[acc_flag] & oracle.FLAG_CUT)
        cdf_flag = next((i for i in range(K + 1) if flags[i] & oracle.FLAG_CDF), None)
        if greedy:
            acc_flag = cdf_flag = None
        rt = ref["tokens"][b]
        if acc_flag is not None:
            i = acc_flag
            if cut:
                rep.cut_flagged += 1
            else:
                rep.acc_flagged += 1
            rep.excluded += K + 1 - i
            if not (g_tok[b, :i] == rt[:i]).all() or g_len[b] < i + 1:
                rep.errors.append((b, "prefix before flagged test at %d differs" % i))
            if g_prob is not None:
                upto = i if cut else i + 1  # a flagged cut may move theta_i itself
                ok = np.abs(g_prob[b, :upto] - ref["accept_prob"][b, :upto]) <= PROB_ATOL
                if i < K and not ok.all():
                    rep.errors.append((b, "accept_prob differs before flagged position"))
            continue
        if g_len[b] != L:
            rep.errors.append((b, "accept_len %d vs oracle %d" % (g_len[b], L)))
            continue
        if cdf_flag is not None:
            n = cdf_flag
            rep.cdf_flagged += 1
            same = np.ones(K + 1, bool)
            same[n] = False
            if not (g_tok[b][same] == rt[same]).all() or not (0 <= g_tok[b, n] < V):
                rep.errors.append((b, "tokens differ outside the flagged draw"))
            elif g_tok[b, n] != rt[n]:
                rep.cdf_differ += 1
                if ref["margins"][b, K] > STRICT_TOL:
                    rep.errors.append((b, "draw differs at margin %.2e > %.0e"
                                       % (ref["margins"][b, K], STRICT_TOL)))
                rep.to_verify.append((b, n, int(g_tok[b, n])))
        elif not (g_tok[b] == rt).all():
            rep.errors.append((b, "tokens %s vs oracle %s" % (g_tok[b].tolist(), rt.tolist())))
        if g_prob is not None and not greedy:
            diff = np.abs(g_prob[b] - ref["accept_prob"][b])
            if not (diff <= PROB_ATOL).all():
                rep.errors.append((b, "accept_prob max diff %.3g" % diff.max()))
    return rep


def verify_draws(wl, rep: SampleReport, temperature=None):
    """Flagged draws where the GPU chose another token than the oracle: the
    GPU token's exact CDF step must come within FLAG_TOL * W of u * W."""
    if not rep.to_verify:
        return
    idx = np.array([b for b, _, _ in rep.to_verify])
    toks = np.array([t for _, _, t in rep.to_verify], np.int32)

    def sub(a):
        return None if a is None else np.ascontiguousarray(a[idx])

    T = wl.T if temperature is None else temperature
    out = oracle.sample(sub(wl.target), sub(wl.draft), sub(wl.draft_tokens), sub(wl.uniforms),
                        T, draft_lens=sub(wl.draft_lens), probe_tokens=toks,
                        token_mask=sub(wl.token_mask), top_k=wl.top_k,
                        top_p=float(np.float32(wl.top_p)))
    u = wl.uniforms[idx, wl.K].astype(np.float64)
    lo, hi = out["probe"][:, 0], out["probe"][:, 1]
    ok = (hi > lo) & (lo <= u + FLAG_TOL) & (hi >= u - FLAG_TOL)
    for j in np.nonzero(~ok)[0]:
        rep.errors.append((int(idx[j]), "GPU draw %d outside the window: step [%.9f, %.9f) u %.9f"
                           % (toks[j], lo[j], hi[j], u[j])))
    rep.to_verify = []


def compare_compaction(gpu, K):
    tok = gpu.tokens.cpu().numpy()
    L = gpu.accept_len.cpu().numpy()
    cu, packed, bid = oracle.compact(tok, L)
    assert (gpu.cu_accept.cpu().numpy() == cu).all(), "cu_accept differs"
    assert (gpu.packed.cpu().numpy() == packed).all(), "packed tokens differ"
    assert (gpu.batch_id.cpu().numpy() == bid).all(), "batch ids differ"


def assert_report(rep: SampleReport, max_flag_rate=None):
    assert not rep.to_verify, "verify_draws() was not run"
    assert not rep.errors, "%d mismatching requests, first: %s" % (len(rep.errors), rep.errors[:5])
    if max_flag_rate is not None:
        assert rep.acc_flagged + rep.cut_flagged <= max_flag_rate * rep.positions, rep.summary()
