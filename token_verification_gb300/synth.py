"""Seeded synthetic inputs for the verification step.

This module is the one piece shared by the tests, the benchmark and the
oracle runs: it draws inputs and nothing else.  It holds none of the
verification arithmetic (no softmax, no acceptance test, no inverse-CDF
draw).  Where a workload needs draft tokens *sampled* from a draft
distribution, they are drawn with the Gumbel-max construction
(argmax of d/T + Gumbel noise), which samples from softmax(d/T) without
computing it; where the proposer is deterministic, drafts come from a plain
argmax or a uniform id, as that proposer would produce them.

Recipe (all draws from numpy's PCG64 streams, seeded per quantity):
  target logits  l = 3 * N(0, 1) + prior[j],  prior[perm[r]] = -1.1 * ln(r + 1)
                 with perm a seeded permutation of the vocabulary (a log-Zipf
                 prior with s = 1.1), then rounded to bfloat16 (round to
                 nearest even) unless the workload is fp32;
  draft logits   d = l + N(0, sigma^2) on the rounded l, rounded the same way;
  draft tokens   dense drafts: Gumbel-max samples of softmax(d / T) taken in
                 float64 from the rounded d; one-hot (n-gram style) drafts: per
                 position with probability p_argmax the argmax of the target
                 row, otherwise a uniform id;
  uniforms       U[0, 1) float32, one per position for the acceptance test and
                 one per request (last column) for the residual / bonus draw;
  tree tokens    children of a node take the top-k ids of a noisy copy
                 (sigma = 0.5) of the node's own target row, in descending
                 order, k = the node's child count;
  n-gram contexts  (the proposer's input) token histories of length
                 U[L/2, L] built from spans of 8..64 tokens: with probability
                 p_copy a copy of an earlier span of the same history (the
                 overlap that code editing and document question answering
                 show), otherwise fresh ids (uniform over the vocabulary);
  grammar masks  (structured output) per position, with probability p_free the
                 grammar allows every token (free text), otherwise a set of
                 round(allowed_frac * V) uniform ids (duplicates merge); packed
                 32 tokens per 32-bit word, token j at bit j % 32 of word
                 j // 32.  Drafts then follow the mask as a grammar-constrained
                 proposer's would: the argmax / Gumbel-max over the allowed
                 tokens, and random ids drawn among the allowed ones.

The standard workloads mirror the vocabularies and draft lengths the pages
use (Llama-3, Qwen, DeepSeek-V3 vocabularies; K = 1..5; batch up to 256);
workload 5 is workload 2 under grammar masks, workload 6 the n-gram proposer
that makes workload 2's kind of drafts, workload 7 workload 2 with top-p
sampling, workloads 8 and 9 typical acceptance on workload 4's tree and on
workload 2's chains, workload 10 lossless tree verification by rejection
sampling on workload 4's tree (uniforms [B, N+1]: node n's test in column n,
the final draw in column 0).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

# name, shapes and draft structure of the five standard workloads
WORKLOADS = {
    0: dict(name="tiny-dense-B4-K3-V1024-fp32", kind="sample", B=4, K=3, V=1024,
            dtype="f32", T=1.0, drafts="dense", sigma=0.7),
    1: dict(name="llama3-vocab-dense-B64-K3-V128256", kind="sample", B=64, K=3, V=128256,
            dtype="bf16", T=0.8, drafts="dense", sigma=0.5),
    2: dict(name="qwen-vocab-onehot-B256-K5-V152064", kind="sample", B=256, K=5, V=152064,
            dtype="bf16", T=1.0, drafts="onehot", p_argmax=0.6),
    3: dict(name="dsv3-vocab-mtp-B128-K1-V129280", kind="sample", B=128, K=1, V=129280,
            dtype="bf16", T=1.0, drafts="dense", sigma=0.25),
    4: dict(name="medusa-tree-B32-N60-V32000", kind="tree", B=32, V=32000, dtype="bf16",
            sigma=0.5, tree="medusa60"),
    # workload 2 under grammar masks (structured output)
    5: dict(name="qwen-vocab-onehot-grammar-B256-K5-V152064", kind="sample", B=256, K=5,
            V=152064, dtype="bf16", T=1.0, drafts="onehot", p_argmax=0.6,
            grammar=dict(p_free=0.3, allowed_frac=0.02)),
    # workload 2 sampled with temperature 0.8 and top_p 0.95
    7: dict(name="qwen-vocab-onehot-topp-B256-K5-V152064", kind="sample", B=256, K=5,
            V=152064, dtype="bf16", T=0.8, drafts="onehot", p_argmax=0.6, top_p=0.95),
    # typical acceptance (Medusa's rule, eps 0.09, delta 0.3): on workload 4's tree and on
    # workload 2's chains
    8: dict(name="medusa-tree-typical-B32-N60-V32000", kind="tree_typical", B=32, V=32000,
            dtype="bf16", sigma=0.5, tree="medusa60", T=1.0, eps=0.09, delta=0.3),
    9: dict(name="qwen-vocab-onehot-typical-B256-K5-V152064", kind="typical", B=256, K=5,
            V=152064, dtype="bf16", T=1.0, drafts="onehot", p_argmax=0.6, eps=0.09, delta=0.3),
    # lossless tree verification by rejection sampling on workload 4's tree
    10: dict(name="medusa-tree-sample-B32-N60-V32000", kind="tree_sample", B=32, V=32000,
             dtype="bf16", sigma=0.5, tree="medusa60", T=1.0),
    # the n-gram proposer that makes workload 2's drafts (prompt_lookup_max 4, K 5)
    6: dict(name="ngram-propose-B256-L4096-V152064", kind="ngram", B=256, K=5, V=152064,
            L=4096, n_min=1, n_max=4),
}


@dataclass
class Workload:
    """Host-side inputs.  Logits are float32 arrays for fp32 workloads and
    uint16 arrays of bfloat16 bit patterns for bf16 workloads."""
    dtype: str
    B: int
    V: int
    target: np.ndarray
    K: int = 0
    T: float = 1.0
    draft: Optional[np.ndarray] = None
    draft_tokens: Optional[np.ndarray] = None
    draft_lens: Optional[np.ndarray] = None
    uniforms: Optional[np.ndarray] = None
    parent: Optional[np.ndarray] = None
    node_tokens: Optional[np.ndarray] = None
    max_depth: int = 0
    token_mask: Optional[np.ndarray] = None  # [B, K+1, ceil(V/32)] uint32
    top_k: int = 0                           # sampling filters (0 / 1.0: off)
    top_p: float = 1.0
    eps: float = 0.0                         # typical acceptance thresholds
    delta: float = 0.0
    history: Optional[np.ndarray] = None     # [B, L] int32 n-gram proposer contexts
    history_lens: Optional[np.ndarray] = None
    meta: dict = field(default_factory=dict)

    def logits_as_float(self, which="target"):
        a = getattr(self, which)
        return bf16_bits_to_float(a) if self.dtype == "bf16" else a


# ---------------------------------------------------------------------------
# elementary draws
# ---------------------------------------------------------------------------

def _rng(seed, *stream):
    return np.random.default_rng([int(seed)] + [int(s) for s in stream])


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (torch's
    conversion)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def zipf_prior(rng, V, s=1.1):
    perm = rng.permutation(V)
    prior = np.empty(V, np.float32)
    prior[perm] = (-s * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)
    return prior


def target_logits(rng, rows, V, scale=3.0):
    """[rows, V] float32: scale * N(0,1) + a log-Zipf prior over a seeded
    permutation of the vocabulary."""
    prior = zipf_prior(rng, V)
    out = rng.standard_normal((rows, V), dtype=np.float32)
    out *= np.float32(scale)
    out += prior[None, :]
    return out


def gumbel_max_tokens(rng, logits_f64, T):
    """One sample per row from softmax(logits / T) by the Gumbel-max
    construction (argmax of logits / T + Gumbel noise)."""
    g = -np.log(-np.log(rng.random(logits_f64.shape)))
    return np.argmax(logits_f64 / T + g, axis=-1).astype(np.int32)


def _finish(x, dtype):
    return round_to_bf16_bits(x) if dtype == "bf16" else np.ascontiguousarray(x, np.float32)


def _as_float(x, dtype):
    return bf16_bits_to_float(x) if dtype == "bf16" else x


def grammar_masks(rng, B, K1, V, p_free=0.3, allowed_frac=0.02, junk_tail=False):
    """[B, K1, ceil(V/32)] uint32 bitmasks (see the recipe above).  Bits past
    V are clear, or random when ``junk_tail`` (they must be ignored)."""
    W = (V + 31) // 32
    words = np.full((B, K1, W), 0xFFFFFFFF, np.uint32)
    constrained = rng.random((B, K1)) >= p_free
    n = max(1, int(round(allowed_frac * V)))
    for b, i in zip(*np.nonzero(constrained)):
        ids = rng.integers(0, V, n)
        row = np.zeros(W, np.uint32)
        np.bitwise_or.at(row, ids >> 5, np.left_shift(np.uint32(1), (ids & 31).astype(np.uint32)))
        words[b, i] = row
    if V % 32:
        tail = np.uint32((1 << (V % 32)) - 1)
        junk = rng.integers(0, 2 ** 32, size=(B, K1), dtype=np.uint64).astype(np.uint32)
        words[..., -1] = (words[..., -1] & tail) | ((junk & ~tail) if junk_tail else np.uint32(0))
    return words


def allowed_tokens(words_row, V):
    """Boolean [V] of the tokens one mask row allows."""
    return np.unpackbits(np.ascontiguousarray(words_row, "<u4").view(np.uint8),
                         bitorder="little")[:V].astype(bool)


# ---------------------------------------------------------------------------
# sampling / greedy workloads
# ---------------------------------------------------------------------------

def make_sample_case(B, K, V, *, dtype="bf16", T=1.0, drafts="dense", sigma=0.5,
                     p_argmax=0.6, seed=0, draft_lens=None, mask_frac=0.0,
                     quantize=None, uniform_seed=None, grammar=None) -> Workload:
    """A verification batch.  ``drafts`` is 'dense' (draft logits given) or
    'onehot' (deterministic proposer, no draft logits).  ``mask_frac`` sets
    that fraction of logits to -inf (never a whole row); ``quantize`` rounds
    logits to multiples of that step (to create exact ties); ``grammar``
    (a dict of grammar_masks keyword arguments) adds grammar masks, with the
    drafts drawn under them."""
    r_l, r_d, r_t, r_m = (_rng(seed, 1), _rng(seed, 2), _rng(seed, 3), _rng(seed, 4))
    r_u = np.random.default_rng(int(seed) if uniform_seed is None else int(uniform_seed))
    tl = target_logits(r_l, B * (K + 1), V)
    if quantize:
        tl = (np.round(tl / quantize) * quantize).astype(np.float32)
    if mask_frac > 0:
        m = r_m.random(tl.shape) < mask_frac
        m[:, 0] = False  # keep one finite logit per row
        tl[m] = -np.inf
    target = _finish(tl, dtype).reshape(B, K + 1, V)
    tf = _as_float(target, dtype)
    draft = None
    if drafts == "dense":
        noise = r_d.standard_normal((B, K, V), dtype=np.float32) * np.float32(sigma)
        dl = tf[:, :K, :] + noise
        draft = _finish(dl, dtype).reshape(B, K, V)
        df = _as_float(draft, dtype).astype(np.float64)
        if T > 0:
            toks = gumbel_max_tokens(r_t, df, T)
        else:
            toks = np.argmax(df, axis=-1).astype(np.int32)
    elif drafts == "onehot":
        take_argmax = r_t.random((B, K)) < p_argmax
        rand_ids = r_t.integers(0, V, size=(B, K), dtype=np.int64).astype(np.int32)
        am = np.argmax(tf[:, :K, :], axis=-1).astype(np.int32) if K > 0 else rand_ids
        toks = np.where(take_argmax, am, rand_ids).astype(np.int32)
    else:
        raise ValueError("drafts must be 'dense' or 'onehot'")
    masks = None
    if grammar is not None:
        r_g = _rng(seed, 5)
        masks = grammar_masks(r_g, B, K + 1, V, **grammar)
        toks = toks.reshape(B, K).copy()
        for b in range(B):
            for i in range(K):
                ok = allowed_tokens(masks[b, i], V)
                if drafts == "dense":
                    g = -np.log(-np.log(r_g.random(V)))
                    score = _as_float(draft[b, i], dtype).astype(np.float64) / (T if T > 0 else 1)
                    toks[b, i] = np.argmax(np.where(ok, score + (g if T > 0 else 0), -np.inf))
                elif take_argmax[b, i]:
                    toks[b, i] = np.argmax(np.where(ok, tf[b, i], -np.inf))
                else:
                    toks[b, i] = r_g.choice(np.nonzero(ok)[0])
    uniforms = r_u.random((B, K + 1), dtype=np.float32)
    lens = None if draft_lens is None else np.ascontiguousarray(draft_lens, np.int32)
    return Workload(dtype=dtype, B=B, V=V, K=K, T=float(T), target=target, draft=draft,
                    draft_tokens=np.ascontiguousarray(toks.reshape(B, K), np.int32),
                    draft_lens=lens, uniforms=uniforms, token_mask=masks,
                    meta=dict(drafts=drafts, sigma=sigma, seed=seed, grammar=grammar))


# ---------------------------------------------------------------------------
# tree workloads
# ---------------------------------------------------------------------------

def medusa60_parent():
    """The 60-node candidate tree: top-3 x top-3 x top-2 x top-1 beneath the
    root in breadth-first order (3 + 9 + 18 + 18 = 48 nodes), plus one
    top-1 child under each of the first 12 depth-4 nodes (nodes 49..60),
    so N = 60 and the depth is 5.  Returns parent[n-1] for n = 1..60."""
    parent = []
    level = [0]
    nid = 1
    for k in (3, 3, 2, 1):
        nxt = []
        for p in level:
            for _ in range(k):
                parent.append(p)
                nxt.append(nid)
                nid += 1
        level = nxt
    for p in level[:12]:
        parent.append(p)
        nid += 1
    return np.asarray(parent, np.int32)


def tree_depths(parent):
    d = [0]
    for n, p in enumerate(parent, start=1):
        d.append(d[p] + 1)
    return np.asarray(d, np.int32)


def make_tree_case(B, V, parent, *, dtype="bf16", sigma=0.5, seed=0, mask_frac=0.0,
                   quantize=None) -> Workload:
    parent = np.asarray(parent, np.int32)
    N = parent.size
    r_l, r_d, r_m = _rng(seed, 11), _rng(seed, 12), _rng(seed, 14)
    tl = target_logits(r_l, B * (N + 1), V)
    if quantize:
        tl = (np.round(tl / quantize) * quantize).astype(np.float32)
    if mask_frac > 0:
        m = r_m.random(tl.shape) < mask_frac
        m[:, 0] = False
        tl[m] = -np.inf
    target = _finish(tl, dtype).reshape(B, N + 1, V)
    tf = _as_float(target, dtype)
    children = [[] for _ in range(N + 1)]
    for n, p in enumerate(parent, start=1):
        children[p].append(n)
    node_tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        for p in range(N + 1):
            ch = children[p]
            if not ch:
                continue
            noisy = tf[b, p].astype(np.float64) + sigma * r_d.standard_normal(V)
            order = np.argsort(-noisy, kind="stable")[: len(ch)]
            for c, tok in zip(ch, order):
                node_tokens[b, c - 1] = tok
    depth = int(tree_depths(parent).max()) if N else 0
    return Workload(dtype=dtype, B=B, V=V, target=target, parent=parent,
                    node_tokens=node_tokens, max_depth=depth,
                    meta=dict(sigma=sigma, seed=seed, N=N))


# ---------------------------------------------------------------------------
# the standard workloads
# ---------------------------------------------------------------------------

def make_workload(index: int, seed: int = 0) -> Workload:
    """The standard workload ``index`` (0..9), seeded by ``seed + index``
    for its uniforms and by (seed + index, stream) for everything else."""
    w = WORKLOADS[index]
    s = seed + index
    if w["kind"] == "ngram":
        ctx = make_ngram_case(w["B"], w["L"], w["V"], seed=s)
        wl = Workload(dtype="int32", B=w["B"], V=w["V"], target=np.empty(0, np.float32),
                      K=w["K"], history=ctx["tokens"], history_lens=ctx["lens"],
                      meta=dict(n_min=w["n_min"], n_max=w["n_max"], L=w["L"]))
    elif w["kind"] in ("tree", "tree_typical", "tree_sample"):
        wl = make_tree_case(w["B"], w["V"], medusa60_parent(), dtype=w["dtype"],
                            sigma=w["sigma"], seed=s)
        if w["kind"] == "tree_typical":  # one uniform per request for the final draw
            wl.uniforms = np.random.default_rng(int(s)).random(w["B"], dtype=np.float32)
        if w["kind"] == "tree_sample":  # node n's test in column n, the final draw in column 0
            wl.uniforms = np.random.default_rng(int(s)).random((w["B"], len(wl.parent) + 1),
                                                              dtype=np.float32)
            wl.T = w["T"]
    else:
        wl = make_sample_case(w["B"], w["K"], w["V"], dtype=w["dtype"], T=w["T"],
                              drafts=w["drafts"], sigma=w.get("sigma", 0.0),
                              p_argmax=w.get("p_argmax", 0.6), seed=s, uniform_seed=s,
                              grammar=w.get("grammar"))
        wl.top_k, wl.top_p = w.get("top_k", 0), w.get("top_p", 1.0)
    if w["kind"] in ("typical", "tree_typical"):
        wl.T, wl.eps, wl.delta = w["T"], w["eps"], w["delta"]
        wl.meta["typical"] = True
    wl.meta["workload"] = w["name"]
    wl.meta["index"] = index
    return wl


# ---------------------------------------------------------------------------
# n-gram proposer inputs
# ---------------------------------------------------------------------------

def make_ngram_case(B, L, V, *, p_copy=0.5, seed=0):
    """Token histories for the prompt-lookup proposer: tokens [B, L] int32
    (entries past lens[b] hold junk ids), lens [B] int32 in [L/2, L]."""
    rng = _rng(seed, 6)
    tokens = rng.integers(0, V, size=(B, L), dtype=np.int64).astype(np.int32)
    lens = rng.integers(max(0, L // 2), L + 1, size=B).astype(np.int32)
    for b in range(B):
        pos = 0
        row = tokens[b]
        while pos < lens[b]:
            span = int(rng.integers(8, 65))
            end = min(pos + span, int(lens[b]))
            if pos >= 8 and rng.random() < p_copy:
                src = int(rng.integers(0, pos - 1))
                for t in range(pos, end):  # element by element: a copy may overlap itself
                    row[t] = row[src + t - pos]
            pos = end
    return dict(tokens=tokens, lens=lens)
