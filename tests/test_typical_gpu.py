"""Typical acceptance on chains and candidate trees: CUDA path vs the fp64
oracle (needs a GPU).  A test the GPU decided differently must be one the
oracle flags (p(x) within 1e-5 of its threshold), and the GPU must then
match the oracle with that test flipped; a final draw may differ from the
oracle's only where the oracle flags it with a margin of at most 1e-6, and
must land in its exact CDF window; p(x) within 1e-5 (tests/parity.py)."""
import numpy as np
import pytest
import torch

import parity
from token_verification_gb300 import api, synth

pytestmark = pytest.mark.gpu
THREADS = 16


def check_chain(wl, eps, delta, d=None, flag_rate=None):
    d = parity.to_device(wl) if d is None else d
    out = api.spec_verify_typical(d["target"], d["draft_tokens"], d["uniforms"], wl.T, eps, delta,
                                  draft_lens=d["draft_lens"])
    torch.cuda.synchronize()
    rep = parity.compare_typical(wl, out, eps, delta, threads=THREADS)
    parity.assert_report(rep, flag_rate)
    return out, rep


@pytest.mark.parametrize("V,K,T,dtype,eps,delta", [
    (152064, 5, 1.0, "bf16", 0.09, 0.3), (32000, 3, 0.7, "bf16", 0.2, 0.5),
    (1025, 4, 1.0, "f32", 0.05, 0.2), (50257, 2, 1.3, "bf16", 0.3, 0.1),
    (9000, 0, 1.0, "bf16", 0.09, 0.3)])
def test_typical_chain(V, K, T, dtype, eps, delta):
    wl = synth.make_sample_case(64, K, V, dtype=dtype, T=T, drafts="onehot", p_argmax=0.7,
                                seed=V + K)
    out, _ = check_chain(wl, eps, delta)
    parity.compare_compaction(out, K)


def test_typical_chain_flag_rate(capsys):
    """Workload 9 at full size and more: flagged tests below 1e-4 of the
    positions, every flagged test and every differing draw verified."""
    total = parity.SampleReport()
    for seed in range(3):
        wl = synth.make_sample_case(256, 5, 152064, drafts="onehot", p_argmax=0.6, seed=200 + seed)
        total.merge(check_chain(wl, 0.09, 0.3)[1])
    with capsys.disabled():
        print("\n[typical chains B256 K5 V152064] %s" % total.summary())
    parity.assert_report(total, max_flag_rate=1e-4)


def test_typical_chain_ragged_and_errors():
    B, K, V = 24, 4, 6000
    lens = np.random.default_rng(4).integers(0, K + 1, size=B).astype(np.int32)
    wl = synth.make_sample_case(B, K, V, drafts="onehot", seed=44, draft_lens=lens)
    tgt = synth.bf16_bits_to_float(wl.target).copy()
    wl.draft_tokens[3, 0] = V
    tgt[5, 0, :] = -np.inf
    tgt[6, 0, 7] = np.nan
    wl.target = synth.round_to_bf16_bits(tgt)
    wl.T = 1.0
    out, _ = check_chain(wl, 0.09, 0.3)
    st = out.status.cpu().numpy()
    assert st[3] == api.REQ_BAD_TOKEN


def check_tree(wl, T, eps, delta, u, parent=None):
    d = parity.to_device(wl)
    par = d["parent"] if parent is None else torch.from_numpy(parent).cuda()
    out = api.spec_verify_tree_typical(d["target"], par, d["node_tokens"],
                                       torch.from_numpy(u).cuda(), T, eps, delta, wl.max_depth)
    torch.cuda.synchronize()
    wl.uniforms = u
    rep = parity.compare_tree(wl, out, "typical", T, eps, delta, threads=THREADS, parent=parent)
    parity.assert_report(rep)
    return out, rep


def test_tree_typical_medusa60():
    wl = synth.make_workload(4)
    u = np.random.default_rng(5).random(wl.B).astype(np.float32)
    for eps, delta in ((0.09, 0.3), (0.3, 0.6), (0.01, 0.05)):
        out, _ = check_tree(wl, 1.0, eps, delta, u)
        assert (out.accept_len.cpu().numpy() >= 2).mean() > 0.3


def test_tree_typical_random_shapes():
    rng = np.random.default_rng(32)
    for trial in range(6):
        N = int(rng.integers(1, 120))
        parent = [int(rng.integers(0, n)) for n in range(1, N + 1)]
        V = int(rng.choice([7, 1000, 32000, 50001]))
        dtype = "f32" if trial % 3 == 0 else "bf16"
        wl = synth.make_tree_case(12, V, parent, dtype=dtype, seed=trial)
        u = rng.random(12).astype(np.float32)
        check_tree(wl, float(rng.choice([0.7, 1.0, 1.5])), 0.1, 0.4, u)


def test_tree_typical_per_request_trees():
    """A parent array per request (device memory), one of them not a tree."""
    rng = np.random.default_rng(34)
    B, N, V = 12, 30, 5000
    parents = np.stack([np.array([int(rng.integers(0, n)) for n in range(1, N + 1)], np.int32)
                        for _ in range(B)])
    parents[4, 6] = 9  # not an earlier node
    wl = synth.make_tree_case(B, V, parents[0], seed=8)
    wl.max_depth = int(max(synth.tree_depths(p).max() for p in np.delete(parents, 4, 0)))
    u = rng.random(B).astype(np.float32)
    out, _ = check_tree(wl, 1.0, 0.2, 0.5, u, parent=parents)
    assert out.status.cpu().numpy()[4] == api.REQ_BAD_TREE
