"""n-gram (prompt-lookup) proposer: CUDA kernel vs the oracle, bit-exact
(needs a GPU).  Contexts come from token_verification_gb300.synth
(make_ngram_case: token histories with copied spans, as in code editing or
document question answering); the edge cases cover empty and one-token
contexts, lengths outside [0, L], a single repeated token, n_min = n_max and
matches that overlap the pattern itself."""
import numpy as np
import pytest
import torch

import oracle
from token_verification_gb300 import api, synth

pytestmark = pytest.mark.gpu


def run(tokens, lens, n_min, n_max, K):
    t = torch.from_numpy(np.ascontiguousarray(tokens, np.int32)).cuda()
    ln = torch.from_numpy(np.ascontiguousarray(lens, np.int32)).cuda()
    out = api.spec_ngram_propose(t, ln, K=K, n_min=n_min, n_max=n_max)
    torch.cuda.synchronize()
    return out


def check(tokens, lens, n_min, n_max, K):
    out = run(tokens, lens, n_min, n_max, K)
    ref = oracle.ngram(tokens, lens, n_min, n_max, K)
    assert (out.draft_lens.cpu().numpy() == ref["draft_lens"]).all()
    assert (out.drafts.cpu().numpy() == ref["drafts"]).all()
    assert (out.match.cpu().numpy() == ref["match"]).all()
    assert (out.status.cpu().numpy() == ref["status"]).all()
    return out, ref


@pytest.mark.parametrize("B,L,V,n_min,n_max,K", [
    (256, 4096, 152064, 1, 4, 5), (64, 700, 50, 1, 4, 5), (32, 20000, 32000, 2, 8, 7),
    (8, 3000, 3, 1, 32, 31), (128, 513, 1000, 4, 4, 1), (16, 9000, 128256, 1, 1, 3)])
def test_ngram_matches_oracle(B, L, V, n_min, n_max, K):
    wl = synth.make_ngram_case(B, L, V, seed=B + L)
    check(wl["tokens"], wl["lens"], n_min, n_max, K)


def test_ngram_edge_cases():
    L = 40
    t = np.zeros((9, L), np.int32)
    lens = np.array([0, 1, 2, L, L, 5, L + 1, -3, 7], np.int32)
    t[2, :2] = [3, 3]                         # one-token repeat
    t[3] = 5                                  # a single repeated token: overlap with itself
    t[4] = np.arange(L) % 7                   # period 7
    t[5, :5] = [1, 2, 1, 2, 1]
    t[8, :7] = [9, 8, 7, 6, 5, 4, 3]          # no repeat at all
    for n_min, n_max, K in ((1, 4, 5), (2, 2, 3), (1, 32, 31), (3, 5, 0)):
        out, ref = check(t, lens, n_min, n_max, K)
    assert list(ref["status"][6:8]) == [oracle.BAD_DRAFT_LEN] * 2


def test_ngram_feeds_onehot_verify():
    """The proposer's drafts and lengths go straight into the one-hot
    verification call as its drafts and draft_lens; the result matches the
    oracle on the same drafts."""
    import parity
    B, L, V, K = 32, 2048, 32000, 5
    ctx = synth.make_ngram_case(B, L, V, seed=5)
    out = run(ctx["tokens"], ctx["lens"], 1, 4, K)
    wl = synth.make_sample_case(B, K, V, drafts="onehot", seed=6)
    wl.draft_tokens = np.ascontiguousarray(out.drafts.clamp(min=0).cpu().numpy())
    wl.draft_lens = out.draft_lens.cpu().numpy()
    assert wl.draft_lens.max() > 0
    d = parity.to_device(wl)
    res = api.spec_verify_sample(d["target"], None, d["draft_tokens"], d["uniforms"], wl.T,
                                 draft_lens=out.draft_lens)
    torch.cuda.synchronize()
    parity.check_sample(wl, res)
