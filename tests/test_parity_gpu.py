"""CUDA path vs the fp64 oracle, through the C ABI (needs a GPU).

Every case draws seeded synthetic inputs (token_verification_gb300.synth),
runs the CUDA kernels through the Python binding of libspecverify, and
compares with the oracle on the same inputs: greedy and tree verification
bit-exactly, rejection sampling token-exactly, with the places the oracle
flags (a uniform within rounding distance of a boundary) verified on the
branch the GPU took (tests/parity.py).  The five standard workloads run at
full size in the launch configuration the benchmark times."""
import numpy as np
import pytest
import torch

import oracle
import parity
from token_verification_gb300 import api, synth

pytestmark = pytest.mark.gpu
THREADS = 16


def run_sample(wl, T=None, **kw):
    d = parity.to_device(wl)
    T = wl.T if T is None else T
    out = api.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], T,
                                 draft_lens=d["draft_lens"], **kw)
    torch.cuda.synchronize()
    return out


def check_sample(wl, T=None, flag_rate=None):
    out = run_sample(wl, T)
    rep = parity.check_sample(wl, out, temperature=T, threads=THREADS, flag_rate=flag_rate)
    parity.compare_compaction(out, wl.K)
    return out, rep


# ---------------------------------------------------------------------------
# the standard workloads at full size
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("index", [0, 1, 2, 3])
def test_standard_workload_sampling(index):
    wl = synth.make_workload(index)
    out, rep = check_sample(wl, flag_rate=1e-4)
    L = out.accept_len.cpu().numpy()
    assert ((L >= 1) & (L <= wl.K + 1)).all()


def test_standard_workload_3_greedy():
    wl = synth.make_workload(3)
    d = parity.to_device(wl)
    out = api.spec_verify_greedy(d["target"], d["draft_tokens"])
    ref = oracle.greedy(wl.target, wl.draft_tokens, threads=THREADS)
    assert (out.tokens.cpu().numpy() == ref["tokens"]).all()
    assert (out.accept_len.cpu().numpy() == ref["accept_len"]).all()
    parity.compare_compaction(out, wl.K)
    # temperature 0 through the sampling entry is the same rule
    out2 = run_sample(wl, T=0.0)
    assert (out2.tokens.cpu().numpy() == ref["tokens"]).all()
    prob = out2.accept_prob.cpu().numpy()
    assert set(np.unique(prob)).issubset({-1.0, 0.0, 1.0})


def test_standard_workload_4_tree():
    wl = synth.make_workload(4)
    d = parity.to_device(wl)
    out = api.spec_verify_tree(d["target"], d["parent"], d["node_tokens"], wl.max_depth)
    ref = oracle.tree(wl.target, wl.parent, wl.node_tokens, wl.max_depth, threads=THREADS)
    for k in ("tokens", "accept_len", "path", "status"):
        assert (getattr(out, k).cpu().numpy() == ref[k]).all(), k
    assert (ref["accept_len"] >= 2).mean() > 0.5  # the workload exercises deep paths


# ---------------------------------------------------------------------------
# edge grid: vocabulary sizes around the chunk and vector widths, K, T, dtype
# ---------------------------------------------------------------------------

GRID = [
    # V, K, T, dtype, drafts
    (1, 2, 1.0, "bf16", "onehot"), (7, 3, 0.8, "f32", "dense"), (8, 1, 1.0, "bf16", "dense"),
    (1000, 5, 2.0, "bf16", "onehot"), (1024, 3, 0.05, "f32", "onehot"),
    (1025, 2, 1.0, "bf16", "dense"), (4104, 4, 0.8, "bf16", "onehot"),
    (32000, 5, 1.0, "bf16", "dense"), (32001, 1, 1.3, "f32", "onehot"),
    (9000, 0, 1.0, "bf16", "onehot"), (5000, 31, 0.9, "bf16", "onehot"),
    (65536, 2, 0.7, "f32", "dense"), (300000, 2, 1.0, "bf16", "dense"),
]


@pytest.mark.parametrize("V,K,T,dtype,drafts", GRID)
def test_sampling_grid(V, K, T, dtype, drafts):
    B = 24
    wl = synth.make_sample_case(B, K, V, dtype=dtype, T=T, drafts=drafts, sigma=0.6, seed=V + K)
    check_sample(wl)


@pytest.mark.parametrize("V,K,dtype", [(1, 1, "bf16"), (7, 3, "f32"), (1000, 5, "bf16"),
                                       (1025, 2, "f32"), (32000, 4, "bf16"), (0 + 129280, 1, "bf16")])
def test_greedy_grid_with_ties(V, K, dtype):
    wl = synth.make_sample_case(16, K, V, dtype=dtype, drafts="onehot", p_argmax=0.8, seed=V,
                                quantize=1.0)  # integer logits: many exact ties
    d = parity.to_device(wl)
    out = api.spec_verify_greedy(d["target"], d["draft_tokens"])
    ref = oracle.greedy(wl.target, wl.draft_tokens)
    assert (out.tokens.cpu().numpy() == ref["tokens"]).all()
    assert (out.accept_len.cpu().numpy() == ref["accept_len"]).all()


def test_ragged_draft_lens():
    B, K, V = 40, 5, 6000
    lens = np.random.default_rng(5).integers(0, K + 1, size=B).astype(np.int32)
    for drafts in ("dense", "onehot"):
        wl = synth.make_sample_case(B, K, V, drafts=drafts, seed=9, draft_lens=lens)
        check_sample(wl)
    wl = synth.make_sample_case(B, K, V, drafts="onehot", p_argmax=0.9, seed=10, draft_lens=lens)
    d = parity.to_device(wl)
    out = api.spec_verify_greedy(d["target"], d["draft_tokens"], draft_lens=d["draft_lens"])
    ref = oracle.greedy(wl.target, wl.draft_tokens, draft_lens=lens)
    assert (out.tokens.cpu().numpy() == ref["tokens"]).all()


def test_masked_logits():
    for drafts in ("dense", "onehot"):
        wl = synth.make_sample_case(32, 3, 20000, drafts=drafts, seed=12, mask_frac=0.5)
        check_sample(wl)


@pytest.mark.parametrize("drafts,V", [("onehot", 4096), ("dense", 4096), ("onehot", 152064)])
def test_flag_rate_many_positions(drafts, V, capsys):
    """Sampling parity over many positions: acceptance tests flagged on fewer
    than 1e-4 of the positions, and each of them verified on the branch the
    GPU took; a draw may differ from the oracle's only where the oracle's
    margin is at most 1e-6 (and then lands in its exact CDF window).  The
    differing draws are reported by the oracle's margin."""
    total = parity.SampleReport()
    B = 2048 if V < 10000 else 256
    for seed in range(10 if V < 10000 else 8):
        wl = synth.make_sample_case(B, 5, V, drafts=drafts, seed=100 + seed)
        out = run_sample(wl)
        total.merge(parity.compare_sample(wl, out, threads=THREADS))
    with capsys.disabled():
        print("\n[flag rate %s V=%d] %s" % (drafts, V, total.summary()))
    parity.assert_report(total, max_flag_rate=1e-4)


def test_data_errors_match_oracle():
    B, K, V = 8, 3, 3000
    wl = synth.make_sample_case(B, K, V, drafts="onehot", seed=21)
    tgt = synth.bf16_bits_to_float(wl.target).copy()
    wl.draft_tokens[1, 0] = V          # token out of range
    wl.draft_tokens[2, 2] = -5
    tgt[3, 0, 17] = np.nan             # NaN in a needed row
    tgt[4, 0, :] = -np.inf             # no finite logit
    tgt[5, 0, 3] = np.inf
    wl.uniforms[6, 0] = 0.999999       # reject at 0 ...
    tgt[6, 2, 5] = np.nan              # ... so the NaN in row 2 is never needed
    wl.target = synth.round_to_bf16_bits(tgt)
    for T in (1.0, 0.0):
        out = run_sample(wl, T=T)
        ref = oracle.sample(wl.target, None, wl.draft_tokens, wl.uniforms, T)
        assert (out.status.cpu().numpy() == ref["status"]).all(), (out.status, ref["status"])
        parity.check_sample(wl, out, temperature=T)
    lens = np.full(B, K, np.int32)
    lens[7] = K + 1
    wl.draft_lens = lens
    out = run_sample(wl)
    assert out.status.cpu().numpy()[7] == api.REQ_BAD_DRAFT_LEN
    assert out.accept_len.cpu().numpy()[7] == 0


def test_tree_random_shapes_and_ties():
    rng = np.random.default_rng(31)
    for trial in range(6):
        N = int(rng.integers(1, 80))
        parent = [int(rng.integers(0, n)) for n in range(1, N + 1)]
        V = int(rng.choice([7, 1000, 1024, 32000, 50001]))
        dtype = "f32" if trial % 3 == 0 else "bf16"
        wl = synth.make_tree_case(12, V, parent, dtype=dtype, seed=trial,
                                  quantize=1.0 if trial % 2 else None)
        d = parity.to_device(wl)
        out = api.spec_verify_tree(d["target"], d["parent"], d["node_tokens"], wl.max_depth)
        ref = oracle.tree(wl.target, wl.parent, wl.node_tokens, wl.max_depth)
        for k in ("tokens", "accept_len", "path", "status"):
            assert (getattr(out, k).cpu().numpy() == ref[k]).all(), (trial, k)


def test_tree_per_request_parents_and_bad_trees():
    """One tree per request in device memory (EAGLE-2's dynamic trees): each
    request's walk follows its own parent array; a request whose array is not
    a tree (a parent that is not an earlier node, or deeper than max_depth)
    gets REQ_BAD_TREE and emits nothing, the others are unaffected."""
    rng = np.random.default_rng(33)
    B, N, V = 16, 40, 6000
    parents = np.stack([np.array([int(rng.integers(0, n)) for n in range(1, N + 1)], np.int32)
                        for _ in range(B)])
    D = int(max(synth.tree_depths(p).max() for p in parents))
    parents[3, 10] = 11                 # a parent after its node
    parents[5, 0] = -1                  # a parent before the root
    wl = synth.make_tree_case(B, V, parents[0], seed=7)
    # node tokens that follow each request's own tree: the top ids of the parent's row
    tf = synth.bf16_bits_to_float(wl.target)
    toks = np.zeros((B, N), np.int32)
    for b in range(B):
        for n in range(1, N + 1):
            pa = parents[b, n - 1] if 0 <= parents[b, n - 1] < n else 0
            order = np.argsort(-tf[b, pa], kind="stable")
            toks[b, n - 1] = order[int(rng.integers(0, 2))]
    wl.node_tokens = toks
    d = parity.to_device(wl)
    par_d = torch.from_numpy(parents).cuda()
    out = api.spec_verify_tree(d["target"], par_d, d["node_tokens"], D)
    ref = oracle.tree(wl.target, parents, toks, D)
    for k in ("tokens", "accept_len", "path", "status"):
        assert (getattr(out, k).cpu().numpy() == ref[k]).all(), k
    st = out.status.cpu().numpy()
    assert st[3] == api.REQ_BAD_TREE and st[5] == api.REQ_BAD_TREE
    assert (ref["accept_len"][st == 0] >= 2).mean() > 0.3
    # a tree deeper than max_depth is a per-request status, not an argument error
    shallow = api.spec_verify_tree(d["target"], par_d, d["node_tokens"], D - 1)
    assert (shallow.status.cpu().numpy() == api.REQ_BAD_TREE).any()


def test_tree_errors():
    wl = synth.make_tree_case(4, 5000, synth.medusa60_parent(), seed=3)
    wl.node_tokens[1, 7] = 5000
    tgt = synth.bf16_bits_to_float(wl.target).copy()
    tgt[2, 0, 9] = np.nan
    wl.target = synth.round_to_bf16_bits(tgt)
    d = parity.to_device(wl)
    out = api.spec_verify_tree(d["target"], d["parent"], d["node_tokens"], wl.max_depth)
    ref = oracle.tree(wl.target, wl.parent, wl.node_tokens, wl.max_depth)
    assert (out.status.cpu().numpy() == ref["status"]).all()
    assert (out.tokens.cpu().numpy() == ref["tokens"]).all()
    short = api.spec_verify_tree(d["target"], d["parent"], d["node_tokens"], wl.max_depth - 1)
    assert (short.status.cpu().numpy() == api.REQ_BAD_TREE).all()
    rc = api._native.lib().spec_verify_tree(  # a parent stride other than 0 or N
        api._p(d["target"]), api._p(d["parent"]), 7, api._p(d["node_tokens"]),
        api._p(out.tokens), api._p(out.accept_len), api.SV_BF16, wl.B, wl.parent.size, wl.V,
        wl.max_depth, None, None, None)
    assert rc == 5  # SV_ERR_TREE


def test_repeatable_and_workspace_reuse():
    """Bit-identical repeat runs (no races), and a workspace shared by calls
    of different shapes stays consistent (every call returns it to zero)."""
    wl_a = synth.make_sample_case(64, 5, 40000, drafts="onehot", seed=41)
    wl_b = synth.make_sample_case(16, 2, 70000, drafts="dense", seed=42)
    outs = []
    for wl in (wl_a, wl_b, wl_a, wl_b, wl_a):
        o = run_sample(wl)
        outs.append((o.tokens.cpu().numpy().copy(), o.accept_prob.cpu().numpy().copy()))
    for i, j in ((0, 2), (2, 4), (1, 3)):
        assert (outs[i][0] == outs[j][0]).all() and (outs[i][1] == outs[j][1]).all()
    parity.check_sample(wl_a, run_sample(wl_a))


def test_empty_batch():
    t = torch.empty((0, 3, 100), dtype=torch.bfloat16, device="cuda")
    dt = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    u = torch.empty((0, 3), dtype=torch.float32, device="cuda")
    out = api.spec_verify_sample(t, None, dt, u, 1.0)
    torch.cuda.synchronize()
    assert out.cu_accept.cpu().tolist() == [0]
