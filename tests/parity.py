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
  * the oracle flags the final draw at position n (u*W within 1e-5 * W of a
    CDF step edge): everything but token n must match; token n is excluded
    (it must still be a valid id).
Greedy and tree verification are compared bit-exactly.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import oracle

PROB_ATOL = 1e-5


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
    return d


def oracle_sample(wl, threads=8, temperature=None):
    T = wl.T if temperature is None else temperature
    return oracle.sample(wl.target, wl.draft, wl.draft_tokens, wl.uniforms, T,
                         draft_lens=wl.draft_lens, threads=threads)


@dataclass
class SampleReport:
    requests: int = 0
    positions: int = 0
    flagged: int = 0
    excluded: int = 0
    errors: list = field(default_factory=list)

    def merge(self, o):
        self.requests += o.requests
        self.positions += o.positions
        self.flagged += o.flagged
        self.excluded += o.excluded
        self.errors += o.errors


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
        acc_flag = next((i for i in range(K + 1) if flags[i] & oracle.FLAG_ACCEPT), None)
        cdf_flag = next((i for i in range(K + 1) if flags[i] & oracle.FLAG_CDF), None)
        if greedy:
            acc_flag = cdf_flag = None
        rt = ref["tokens"][b]
        if acc_flag is not None:
            i = acc_flag
            rep.flagged += 1
            rep.excluded += K + 1 - i
            if not (g_tok[b, :i] == rt[:i]).all() or g_len[b] < i + 1:
                rep.errors.append((b, "prefix before flagged test at %d differs" % i))
            if g_prob is not None:
                ok = np.abs(g_prob[b, :i + 1] - ref["accept_prob"][b, :i + 1]) <= PROB_ATOL
                if i < K and not ok.all():
                    rep.errors.append((b, "accept_prob differs before flagged position"))
            continue
        if g_len[b] != L:
            rep.errors.append((b, "accept_len %d vs oracle %d" % (g_len[b], L)))
            continue
        if cdf_flag is not None:
            n = cdf_flag
            rep.flagged += 1
            rep.excluded += 1
            same = np.ones(K + 1, bool)
            same[n] = False
            if not (g_tok[b][same] == rt[same]).all() or not (0 <= g_tok[b, n] < V):
                rep.errors.append((b, "tokens differ outside the flagged draw"))
        elif not (g_tok[b] == rt).all():
            rep.errors.append((b, "tokens %s vs oracle %s" % (g_tok[b].tolist(), rt.tolist())))
        if g_prob is not None and not greedy:
            diff = np.abs(g_prob[b] - ref["accept_prob"][b])
            if not (diff <= PROB_ATOL).all():
                rep.errors.append((b, "accept_prob max diff %.3g" % diff.max()))
    return rep


def compare_compaction(gpu, K):
    tok = gpu.tokens.cpu().numpy()
    L = gpu.accept_len.cpu().numpy()
    cu, packed, bid = oracle.compact(tok, L)
    assert (gpu.cu_accept.cpu().numpy() == cu).all(), "cu_accept differs"
    assert (gpu.packed.cpu().numpy() == packed).all(), "packed tokens differ"
    assert (gpu.batch_id.cpu().numpy() == bid).all(), "batch ids differ"


def assert_report(rep: SampleReport, max_flag_rate=None):
    assert not rep.errors, "%d mismatching requests, first: %s" % (len(rep.errors), rep.errors[:5])
    if max_flag_rate is not None:
        assert rep.flagged <= max_flag_rate * rep.positions, (
            "flagged %d of %d positions" % (rep.flagged, rep.positions))
