"""Grammar-constrained verification: CUDA path vs the fp64 oracle (needs a
GPU).  The masks come from token_verification_gb300.synth.grammar_masks;
drafts are drawn under them as a grammar-constrained proposer would.  The
cases cover both ways the mask words reach the kernels (bulk-copied with the
logits when the rows are 16-byte aligned, read word by word otherwise), the
scalar path, dense and one-hot drafts, greedy, junk bits past V, and rows
the mask leaves without a finite logit."""
import numpy as np
import pytest
import torch

import oracle
import parity
from token_verification_gb300 import api, synth

pytestmark = pytest.mark.gpu
THREADS = 16


def run_masked(wl, d=None, T=None, mask=None):
    d = parity.to_device(wl) if d is None else d
    T = wl.T if T is None else T
    out = api.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], T,
                                 draft_lens=d["draft_lens"],
                                 token_mask=d["token_mask"] if mask is None else mask)
    torch.cuda.synchronize()
    return out


def check_masked(wl, T=None, d=None, mask=None):
    out = run_masked(wl, d, T, mask)
    parity.check_sample(wl, out, temperature=T, threads=THREADS)
    parity.compare_compaction(out, wl.K)
    # nothing the mask rules out is ever emitted
    toks = out.tokens.cpu().numpy()
    for b in range(wl.B):
        for i in range(wl.K + 1):
            if toks[b, i] >= 0:
                assert synth.allowed_tokens(wl.token_mask[b, i], wl.V)[toks[b, i]], (b, i)
    return out


GRID = [
    # V, K, T, dtype, drafts  (ceil(V/32) % 4 == 0 and V % vec == 0: bulk-copied words)
    (1000, 3, 1.0, "bf16", "onehot"),     # 32 words: bulk
    (4104, 4, 0.8, "bf16", "dense"),      # 129 words: word by word
    (32001, 2, 1.3, "f32", "onehot"),     # scalar path
    (65536, 2, 0.7, "f32", "dense"),      # fp32 vector path, bulk
    (129280, 1, 1.0, "bf16", "dense"),    # 4040 words: bulk
    (50257, 3, 1.0, "bf16", "onehot"),    # scalar path, odd vocabulary
    (30, 2, 1.0, "bf16", "dense"),        # one partial word
]


@pytest.mark.parametrize("V,K,T,dtype,drafts", GRID)
def test_masked_sampling_grid(V, K, T, dtype, drafts):
    wl = synth.make_sample_case(24, K, V, dtype=dtype, T=T, drafts=drafts, sigma=0.6,
                                seed=V + 3 * K, grammar=dict(p_free=0.3, allowed_frac=0.03,
                                                             junk_tail=True))
    check_masked(wl)


@pytest.mark.parametrize("allowed_frac,drafts", [(0.125, "onehot"), (0.125, "dense"),
                                                 (0.0005, "onehot")])
def test_masked_sparse_and_dense_chunks(allowed_frac, drafts):
    """Chunks whose mask allows at most 128 tokens take the streaming
    kernel's sparse path, the others the dense one: at an allowed fraction
    of 1/8 (about 128 per 1024-token chunk) the rows mix both; at 0.0005 most
    chunks allow none or one token."""
    wl = synth.make_sample_case(24, 3, 152064, drafts=drafts, T=0.9, sigma=0.5, seed=82,
                                grammar=dict(p_free=0.2, allowed_frac=allowed_frac,
                                             junk_tail=True))
    check_masked(wl)


@pytest.mark.parametrize("V,dtype", [(1000, "bf16"), (4104, "bf16"), (32001, "f32"),
                                     (152064, "bf16")])
def test_masked_greedy(V, dtype):
    wl = synth.make_sample_case(32, 4, V, dtype=dtype, drafts="onehot", p_argmax=0.8, seed=V,
                                quantize=1.0, grammar=dict(p_free=0.2, allowed_frac=0.05,
                                                           junk_tail=True))
    d = parity.to_device(wl)
    out = api.spec_verify_greedy(d["target"], d["draft_tokens"], token_mask=d["token_mask"])
    ref = oracle.greedy(wl.target, wl.draft_tokens, token_mask=wl.token_mask)
    assert (out.tokens.cpu().numpy() == ref["tokens"]).all()
    assert (out.accept_len.cpu().numpy() == ref["accept_len"]).all()
    parity.compare_compaction(out, wl.K)
    out2 = run_masked(wl, d, T=0.0)  # temperature 0 through the sampling entry
    assert (out2.tokens.cpu().numpy() == ref["tokens"]).all()


def test_masked_headline_shape():
    """B=256, K=5, V=152064 one-hot drafts under grammar masks, full size."""
    wl = synth.make_sample_case(256, 5, 152064, drafts="onehot", seed=77,
                                grammar=dict(p_free=0.3, allowed_frac=0.02))
    check_masked(wl)


def test_masked_dense_cluster_residual():
    """Dense drafts at B=64, V=128256: the residual row pair is read by a
    cluster of CTAs per request, with the mask applied in every chunk."""
    wl = synth.make_sample_case(64, 3, 128256, drafts="dense", T=0.8, sigma=0.5, seed=78,
                                grammar=dict(p_free=0.5, allowed_frac=0.1))
    check_masked(wl)


def test_mask_words_read_one_by_one():
    """The same inputs with the mask rows at a 4-byte (not 16-byte) offset:
    the kernels read the words directly instead of bulk-copying them, with
    identical results."""
    wl = synth.make_sample_case(32, 3, 8192, drafts="onehot", seed=79,
                                grammar=dict(p_free=0.3, allowed_frac=0.05))
    d = parity.to_device(wl)
    flat = torch.zeros(wl.token_mask.size + 1, dtype=torch.int32, device="cuda")
    shifted = flat[1:].view(wl.token_mask.shape)
    shifted.copy_(d["token_mask"])
    assert shifted.data_ptr() % 16 != 0
    a = run_masked(wl, d)
    b = run_masked(wl, d, mask=shifted)
    for k in ("tokens", "accept_len", "accept_prob"):
        assert torch.equal(getattr(a, k), getattr(b, k)), k
    check_masked(wl, d=d, mask=shifted)


def test_mask_edge_cases():
    """A draft outside its mask is rejected even at u = 0; a needed row whose
    mask leaves no finite logit is a data error; an all-ones mask gives the
    unmasked result."""
    B, K, V = 6, 3, 3000
    wl = synth.make_sample_case(B, K, V, drafts="onehot", seed=80,
                                grammar=dict(p_free=0.0, allowed_frac=0.05))
    m = wl.token_mask
    x = wl.draft_tokens
    # request 0: draft 0 ruled out by its mask, u_0 = 0
    m[0, 0, x[0, 0] >> 5] &= ~np.uint32(1 << (x[0, 0] & 31))
    wl.uniforms[0, 0] = 0.0
    # request 1: the mask of position 1 allows only tokens whose logit is -inf
    tgt = synth.bf16_bits_to_float(wl.target).copy()
    allowed = synth.allowed_tokens(m[1, 1], V)
    tgt[1, 1, allowed] = -np.inf
    wl.uniforms[1, 0] = 0.0
    m[1, 0] = 0xFFFFFFFF
    # request 2: a mask that allows nothing at the bonus position
    m[2, K] = 0
    wl.uniforms[2, :K] = 0.0
    m[2, :K] = 0xFFFFFFFF
    # drafts that pass the greedy rule too where the case needs acceptance
    x[1, 0] = np.argmax(tgt[1, 0])
    x[2, :] = np.argmax(tgt[2, :K], axis=-1)
    wl.target = synth.round_to_bf16_bits(tgt)
    for T in (1.0, 0.0):
        out = check_masked(wl, T=T)
        st = out.status.cpu().numpy()
        ref = oracle.sample(wl.target, wl.draft, wl.draft_tokens, wl.uniforms, T,
                            token_mask=wl.token_mask)
        assert (st == ref["status"]).all(), (st, ref["status"])
        assert st[1] == api.REQ_BAD_LOGITS and st[2] == api.REQ_BAD_LOGITS
        assert out.accept_len.cpu().numpy()[0] == 1
    # all-ones masks: identical to the unmasked call
    wl2 = synth.make_sample_case(16, 3, 20000, drafts="dense", seed=81)
    d2 = parity.to_device(wl2)
    ones = torch.full((16, 4, (20000 + 31) // 32), -1, dtype=torch.int32, device="cuda")
    a = run_masked(wl2, d2, mask=ones)
    b = api.spec_verify_sample(d2["target"], d2["draft"], d2["draft_tokens"], d2["uniforms"],
                               wl2.T)
    torch.cuda.synchronize()
    for k in ("tokens", "accept_len", "accept_prob"):
        assert torch.equal(getattr(a, k), getattr(b, k)), k
