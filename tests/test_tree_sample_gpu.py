"""Lossless tree verification by rejection sampling: CUDA path vs the fp64
oracle (needs a GPU).

Candidates are one-hot drafts of the distribution at their parent; the
children of the current node are tested in increasing id against the
residual, a rejected child's token leaves it, and with no child accepted one
token is drawn from the residual ("推测解码与 MTP" §10.4 with the candidate
trees of §3.3 / §4.2).  Paths and tokens must match the oracle exactly; a
node test the GPU decided differently must be one the oracle flags, and the
GPU must then match the oracle with it flipped; a differing final draw must
be flagged within 1e-6 and land in its exact CDF window (tests/parity.py)."""
import numpy as np
import pytest
import torch

import oracle
import parity
from token_verification_gb300 import api, synth

pytestmark = pytest.mark.gpu
THREADS = 16


def run_tree_sample(wl, T, parent=None):
    d = parity.to_device(wl)
    par = d["parent"] if parent is None else torch.from_numpy(parent).cuda()
    out = api.spec_verify_tree_sample(d["target"], par, d["node_tokens"], d["uniforms"], T,
                                      wl.max_depth)
    torch.cuda.synchronize()
    return out


def check_tree_sample(wl, T, parent=None):
    out = run_tree_sample(wl, T, parent)
    rep = parity.compare_tree(wl, out, "sample", T, threads=THREADS, parent=parent)
    parity.assert_report(rep)
    return out, rep


def with_uniforms(wl, seed):
    N = wl.node_tokens.shape[1]
    wl.uniforms = np.random.default_rng(seed).random((wl.B, N + 1), dtype=np.float32)
    return wl


def test_standard_workload_10(capsys):
    """The Medusa-60 tree at full size (B32, V32000), three uniform draws."""
    total = parity.SampleReport()
    for seed in range(3):
        wl = with_uniforms(synth.make_workload(10), 300 + seed)
        out, rep = check_tree_sample(wl, 1.0)
        total.merge(rep)
        L = out.accept_len.cpu().numpy()
        assert ((L >= 1) & (L <= wl.max_depth + 1)).all()
    with capsys.disabled():
        print("\n[tree sampling B32 N60 V32000] %s" % total.summary())


@pytest.mark.parametrize("trial", range(8))
def test_random_trees(trial):
    """Random trees up to 200 nodes; vocabularies around the chunk and
    vector widths (scalar path for odd V), fp32 and bf16, temperatures,
    repeated sibling tokens and tokens of zero probability."""
    rng = np.random.default_rng(40 + trial)
    N = int(rng.integers(1, 200 if trial % 2 else 60))
    parent = [int(rng.integers(0, n)) for n in range(1, N + 1)]
    V = int(rng.choice([5, 1000, 1025, 32000, 50001]))
    dtype = "f32" if trial % 3 == 0 else "bf16"
    T = float(rng.choice([0.6, 1.0, 1.4]))
    wl = synth.make_tree_case(16, V, parent, dtype=dtype, seed=trial, mask_frac=0.2 * (trial % 2))
    toks = wl.node_tokens
    for b in range(16):  # repeat a sibling's token here and there
        for n in range(2, N + 1):
            sib = [c for c in range(1, n) if parent[c - 1] == parent[n - 1]]
            if sib and rng.random() < 0.1:
                toks[b, n - 1] = toks[b, sib[0] - 1]
    with_uniforms(wl, trial)
    check_tree_sample(wl, T)


def test_chain_tree_matches_onehot_chain():
    """A chain-shaped tree is one-hot chain verification: the GPU's tree
    sampler and its one-hot chain call give the same tokens on the same
    logits, with the uniforms remapped (node n's test is chain column n-1,
    the final draw column K)."""
    B, N, V = 64, 5, 40000
    wl = synth.make_tree_case(B, V, list(range(N)), seed=11)
    with_uniforms(wl, 12)
    out = run_tree_sample(wl, 0.9)
    d = parity.to_device(wl)
    u_chain = np.concatenate([wl.uniforms[:, 1:], wl.uniforms[:, :1]], axis=1)
    chain = api.spec_verify_sample(d["target"], None, d["node_tokens"],
                                   torch.from_numpy(np.ascontiguousarray(u_chain)).cuda(), 0.9)
    torch.cuda.synchronize()
    assert torch.equal(out.tokens, chain.tokens)
    assert torch.equal(out.accept_len, chain.accept_len)
    parity.assert_report(parity.compare_tree(wl, out, "sample", 0.9, threads=THREADS))


def test_per_request_trees_and_errors():
    """One tree per request in device memory; a parent array that is not a
    tree, a token outside the vocabulary and a NaN on the walked path are
    per-request statuses, matching the oracle; T = 0 is the greedy walk."""
    rng = np.random.default_rng(50)
    B, N, V = 12, 24, 7000
    parents = np.stack([np.array([int(rng.integers(0, n)) for n in range(1, N + 1)], np.int32)
                        for _ in range(B)])
    parents[2, 5] = 6                   # node 6 (index 5) its own parent
    wl = synth.make_tree_case(B, V, parents[0], seed=13)
    wl.max_depth = int(max(synth.tree_depths(p).max() for p in np.delete(parents, 2, 0)))
    wl.node_tokens[4, 3] = V            # a token outside the vocabulary
    tgt = synth.bf16_bits_to_float(wl.target).copy()
    tgt[6, 0, 11] = np.nan              # the root row is always walked
    wl.target = synth.round_to_bf16_bits(tgt)
    with_uniforms(wl, 14)
    out, _ = check_tree_sample(wl, 1.0, parent=parents)
    st = out.status.cpu().numpy()
    assert st[2] == api.REQ_BAD_TREE and st[4] == api.REQ_BAD_TOKEN
    assert st[6] == api.REQ_BAD_LOGITS
    # temperature 0: the greedy tree walk
    d = parity.to_device(wl)
    g = api.spec_verify_tree_sample(d["target"], torch.from_numpy(parents).cuda(),
                                    d["node_tokens"], d["uniforms"], 0.0, wl.max_depth)
    ref = oracle.tree(wl.target, parents, wl.node_tokens, wl.max_depth)
    for k in ("tokens", "accept_len", "path", "status"):
        assert (getattr(g, k).cpu().numpy() == ref[k]).all(), k


def test_repeatable():
    wl = with_uniforms(synth.make_workload(10), 60)
    a = run_tree_sample(wl, 1.0)
    b = run_tree_sample(wl, 1.0)
    for k in ("tokens", "accept_len", "path", "status"):
        assert torch.equal(getattr(a, k), getattr(b, k)), k
