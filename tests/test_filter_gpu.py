"""Top-k / top-p filtered verification: CUDA path vs the fp64 oracle (needs
a GPU).  Each row of a filtered call is taken by one CTA, which finds the cut
among the row's candidates (elements within 2^-18 of the max's weight) or,
when the cut may lie outside them, by a radix descent over the whole row.
The GPU reports every row's cut value; the oracle runs with those cuts
forced and each must be the rule's own cut or lie within 1e-6 of mass of it
(tests/parity.py).  The cases cover both logit types, the vector and the
scalar row loads, exact ties at the cuts (quantised logits), dense and
one-hot drafts, grammar masks together with the filters, ragged drafts, the
switches (top_k >= V, top_p = 1), and the argument checks."""
import numpy as np
import pytest
import torch

import parity
from token_verification_gb300 import api, synth

pytestmark = pytest.mark.gpu
THREADS = 16


def check_filtered(wl, flag_rate=None):
    d = parity.to_device(wl)
    out = api.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], wl.T,
                                 draft_lens=d["draft_lens"], token_mask=d["token_mask"],
                                 top_k=wl.top_k, top_p=wl.top_p, cut=True)
    torch.cuda.synchronize()
    rep = parity.check_sample(wl, out, threads=THREADS, flag_rate=flag_rate)
    parity.compare_compaction(out, wl.K)
    return out, rep


GRID = [
    # V, K, T, dtype, drafts, top_k, top_p, quantize
    (152064, 3, 0.8, "bf16", "onehot", 0, 0.95, None),   # the cut among the candidates
    (152064, 2, 1.0, "bf16", "dense", 50, 0.9, None),
    (32000, 5, 0.7, "bf16", "onehot", 20, 1.0, 1.0),      # ties at the top-k cut
    (32000, 3, 1.0, "bf16", "dense", 0, 0.8, 0.5),        # ties at the top-p cut
    (65536, 2, 1.3, "f32", "dense", 100, 0.95, None),     # fp32: 4 radix passes
    (50257, 3, 0.9, "bf16", "onehot", 0, 0.9, None),      # scalar row loads (odd V)
    (1000, 4, 1.0, "bf16", "dense", 1, 1.0, None),        # top-k = 1
    (4104, 2, 0.6, "f32", "onehot", 7, 0.3, 0.25),
    (260000, 1, 1.0, "bf16", "onehot", 0, 0.99, None),    # the widest rows (508 KB)
    (9000, 0, 1.0, "bf16", "onehot", 0, 0.5, None),       # K = 0: only the bonus draw
    # rows whose cut may lie outside the candidates (weights >= 2^-18 of the
    # max's) take the full-row radix descent: top-p too close to 1, top-k
    # above the candidate count
    (32000, 3, 1.0, "bf16", "dense", 0, 0.9999, None),
    (32000, 2, 0.3, "bf16", "onehot", 20000, 1.0, None),
    (65536, 2, 0.5, "f32", "onehot", 30000, 0.9, None),
    # nearly every element within 2^-18 of the max's weight: the candidate
    # stages fill up and the rows take the full-row path
    (152064, 2, 2.0, "bf16", "onehot", 0, 0.9, None),
]


@pytest.mark.parametrize("V,K,T,dtype,drafts,top_k,top_p,quantize", GRID)
def test_filtered_grid(V, K, T, dtype, drafts, top_k, top_p, quantize):
    wl = synth.make_sample_case(24, K, V, dtype=dtype, T=T, drafts=drafts, sigma=0.6,
                                seed=V + K + top_k, quantize=quantize)
    wl.top_k, wl.top_p = top_k, top_p
    check_filtered(wl)


def test_filtered_with_grammar_masks_and_ragged_drafts():
    B, K, V = 40, 4, 20000
    lens = np.random.default_rng(3).integers(0, K + 1, size=B).astype(np.int32)
    for drafts in ("onehot", "dense"):
        wl = synth.make_sample_case(B, K, V, drafts=drafts, seed=33, draft_lens=lens, T=0.9,
                                    grammar=dict(p_free=0.3, allowed_frac=0.2))
        wl.top_k, wl.top_p = 40, 0.9
        check_filtered(wl)


def test_filtered_headline_shape(capsys):
    """B=256, K=5, V=152064 one-hot drafts sampled with temperature 0.8 and
    top_p 0.95 (the vLLM Ascend guide's SamplingParams), full size: flagged
    acceptance tests below 1e-4 of the positions, every cut the rule's own
    or within 1e-6 of mass of it (counted), everything after it exact."""
    wl = synth.make_sample_case(256, 5, 152064, drafts="onehot", T=0.8, seed=90)
    wl.top_p = 0.95
    _, rep = check_filtered(wl, flag_rate=1e-4)
    with capsys.disabled():
        print("\n[top-p 0.95, B256 K5 V152064] %s" % rep.summary())


def test_filter_switches_and_argument_checks():
    wl = synth.make_sample_case(16, 3, 5000, drafts="dense", seed=91)
    d = parity.to_device(wl)
    plain = api.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], 1.0)
    off = api.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], 1.0,
                                 top_k=5000, top_p=1.0)
    torch.cuda.synchronize()
    for k in ("tokens", "accept_len", "accept_prob"):
        assert torch.equal(getattr(plain, k), getattr(off, k)), k
    for bad in (dict(top_k=-1), dict(top_p=0.0), dict(top_p=1.5), dict(top_p=float("nan"))):
        with pytest.raises(api.VerifyError):
            api.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], 1.0,
                                   **bad)
    big = torch.zeros((2, 2, 140000), dtype=torch.float32, device="cuda")  # > 512 KB per row
    with pytest.raises(api.VerifyError):
        api.spec_verify_sample(big, None, torch.zeros((2, 1), dtype=torch.int32, device="cuda"),
                               torch.zeros((2, 2), dtype=torch.float32, device="cuda"), 1.0,
                               top_p=0.9)


@pytest.mark.parametrize("T,top_k,top_p", [(0.8, 0, 0.95), (1.0, 40, 0.9), (2.0, 0, 0.9)])
def test_filtered_repeatable(T, top_k, top_p):
    """The cut and the records come from integer (fixed-point) histograms and
    fixed-order sums, so a repeated call gives identical outputs whatever the
    order of the shared-memory atomics: the candidate path (T 0.8), top-k then
    top-p among the candidates, and the full-row path (T 2: the candidate
    stages fill up)."""
    wl = synth.make_sample_case(24, 3, 152064, drafts="onehot", T=T, seed=93)
    d = parity.to_device(wl)
    outs = [api.spec_verify_sample(d["target"], None, d["draft_tokens"], d["uniforms"], T,
                                   top_k=top_k, top_p=top_p) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        for k in ("tokens", "accept_len", "accept_prob"):
            assert torch.equal(getattr(outs[0], k), getattr(o, k)), k
