"""Typical acceptance on chains and candidate trees: CUDA path vs the fp64
oracle (needs a GPU).  A position whose test the oracle flags (p(x) within
1e-5 of its threshold) ends the comparison of its request there (either
outcome is valid); a final draw the oracle flags near a CDF step may pick the
neighbouring token; everything else must match exactly, with p(x) to 1e-5."""
import numpy as np
import pytest
import torch

import oracle
import parity
from token_verification_gb300 import api, synth

pytestmark = pytest.mark.gpu
THREADS = 16
PROB_ATOL = 1e-5


def compare_chain(ref, out, K):
    g_tok, g_len = out.tokens.cpu().numpy(), out.accept_len.cpu().numpy()
    g_st, g_prob = out.status.cpu().numpy(), out.accept_prob.cpu().numpy()
    errors, flagged = [], 0
    for b in range(g_tok.shape[0]):
        if g_st[b] != ref["status"][b]:
            errors.append((b, "status"))
            continue
        if ref["status"][b]:
            continue
        fl = ref["flags"][b]
        acc = next((i for i in range(K + 1) if fl[i] & oracle.FLAG_ACCEPT), None)
        if acc is not None:
            flagged += 1
            if not (g_tok[b, :acc] == ref["tokens"][b, :acc]).all():
                errors.append((b, "prefix before a flagged test"))
            continue
        L = int(ref["accept_len"][b])
        if g_len[b] != L:
            errors.append((b, "accept_len %d vs %d" % (g_len[b], L)))
            continue
        same = g_tok[b] == ref["tokens"][b]
        if not same[:L - 1].all() or (not same[L - 1] and not fl[L - 1] & oracle.FLAG_CDF):
            errors.append((b, "tokens %s vs %s" % (g_tok[b].tolist(), ref["tokens"][b].tolist())))
        tested = ref["accept_prob"][b] >= 0
        if not (np.abs(g_prob[b] - ref["accept_prob"][b])[tested] <= PROB_ATOL).all():
            errors.append((b, "p(x)"))
    assert not errors, errors[:5]
    return flagged


@pytest.mark.parametrize("V,K,T,dtype,eps,delta", [
    (152064, 5, 1.0, "bf16", 0.09, 0.3), (32000, 3, 0.7, "bf16", 0.2, 0.5),
    (1025, 4, 1.0, "f32", 0.05, 0.2), (50257, 2, 1.3, "bf16", 0.3, 0.1),
    (9000, 0, 1.0, "bf16", 0.09, 0.3)])
def test_typical_chain(V, K, T, dtype, eps, delta):
    wl = synth.make_sample_case(64, K, V, dtype=dtype, T=T, drafts="onehot", p_argmax=0.7,
                                seed=V + K)
    d = parity.to_device(wl)
    out = api.spec_verify_typical(d["target"], d["draft_tokens"], d["uniforms"], T, eps, delta)
    torch.cuda.synchronize()
    ref = oracle.typical(wl.target, wl.draft_tokens, wl.uniforms, T, eps, delta, threads=THREADS)
    compare_chain(ref, out, K)
    parity.compare_compaction(out, K)


def test_typical_chain_ragged_and_errors():
    B, K, V = 24, 4, 6000
    lens = np.random.default_rng(4).integers(0, K + 1, size=B).astype(np.int32)
    wl = synth.make_sample_case(B, K, V, drafts="onehot", seed=44, draft_lens=lens)
    tgt = synth.bf16_bits_to_float(wl.target).copy()
    wl.draft_tokens[3, 0] = V
    tgt[5, 0, :] = -np.inf
    tgt[6, 0, 7] = np.nan
    wl.target = synth.round_to_bf16_bits(tgt)
    d = parity.to_device(wl)
    out = api.spec_verify_typical(d["target"], d["draft_tokens"], d["uniforms"], 1.0, 0.09, 0.3,
                                  draft_lens=d["draft_lens"])
    torch.cuda.synchronize()
    ref = oracle.typical(wl.target, wl.draft_tokens, wl.uniforms, 1.0, 0.09, 0.3, draft_lens=lens)
    compare_chain(ref, out, K)


def check_tree(wl, T, eps, delta, u):
    d = parity.to_device(wl)
    ut = torch.from_numpy(u).cuda()
    out = api.spec_verify_tree_typical(d["target"], wl.parent, d["node_tokens"], ut, T, eps, delta,
                                       wl.max_depth)
    torch.cuda.synchronize()
    ref = oracle.tree_typical(wl.target, wl.parent, wl.node_tokens, u, T, eps, delta,
                              wl.max_depth, threads=THREADS)
    g = {k: getattr(out, k).cpu().numpy() for k in ("tokens", "accept_len", "path", "status")}
    compared = 0
    for b in range(wl.B):
        assert g["status"][b] == ref["status"][b], b
        if ref["flags"][b] & oracle.FLAG_ACCEPT:
            continue
        compared += 1
        L = int(ref["accept_len"][b])
        assert g["accept_len"][b] == L, (b, g["accept_len"][b], L)
        assert (g["path"][b] == ref["path"][b]).all(), b
        same = g["tokens"][b] == ref["tokens"][b]
        assert same[:max(L - 1, 0)].all(), b
        assert same[L - 1] or ref["flags"][b] & oracle.FLAG_CDF or L == 0, b
    return compared


def test_tree_typical_medusa60():
    wl = synth.make_workload(4)
    u = np.random.default_rng(5).random(wl.B).astype(np.float32)
    for eps, delta in ((0.09, 0.3), (0.3, 0.6), (0.01, 0.05)):
        assert check_tree(wl, 1.0, eps, delta, u) > wl.B // 2


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
