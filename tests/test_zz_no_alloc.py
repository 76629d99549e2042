"""The allocation-free entry point, spec_verify_sample_noalloc.

Callers that cannot allocate device memory (a runtime that keeps the whole
device in its own pool and gives a plugin only its input and output buffers,
or a path where a cudaMalloc and the device synchronisation it may cause are
not allowed) use this entry point: its scratch is a fixed array inside the
library.  The GPU test calls it through the C ABI twice in a row and checks
each result against spec_verify_sample with a caller-provided workspace
(tokens, accept lengths, packed output and statuses identical, accept
probabilities within 1e-5) and against the fp64 oracle under the same rule
as every other sampling test.  This file is collected last so that a run
that stops at the first failure has run every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

import parity
from token_verification_gb300 import _native, api, build, synth


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_rejects_problems_larger_than_the_scratch():
    """No GPU needed: the size check comes before any CUDA call."""
    build.build()
    lib = _native.lib()
    fake = ctypes.c_void_p(0x10000)
    assert lib.spec_verify_workspace_size(4096, 31, 152064) > (8 << 20)
    rc = lib.spec_verify_sample_noalloc(fake, None, fake, fake, ctypes.c_float(1.0), fake, fake,
                                        1, 4096, 31, 152064, None, None, None, None, None, None,
                                        None)
    assert rc == 6  # SV_ERR_WORKSPACE: the fixed scratch is too small


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_point_on_two_calls():
    lib = _native.lib()
    cases = [synth.make_sample_case(64, 5, 32000, drafts="onehot", seed=71),
             synth.make_sample_case(48, 3, 50000, drafts="dense", T=0.8, seed=72)]
    for wl in cases:  # two calls in a row, different shapes and modes
        d = parity.to_device(wl)
        B, K, V = wl.B, wl.K, wl.V
        ref = api.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                                     wl.T)
        out = api.alloc_outputs(B, K, d["target"].device)
        rc = lib.spec_verify_sample_noalloc(
            _p(d["target"]), _p(d["draft"]), _p(d["draft_tokens"]), _p(d["uniforms"]),
            ctypes.c_float(wl.T), _p(out.tokens), _p(out.accept_len), api.SV_BF16, B, K, V, None,
            _p(out.cu_accept), _p(out.packed), _p(out.batch_id), _p(out.accept_prob),
            _p(out.status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0
        torch.cuda.synchronize()
        for name in ("tokens", "accept_len", "cu_accept", "packed", "batch_id", "status"):
            assert torch.equal(getattr(out, name), getattr(ref, name)), name
        diff = (out.accept_prob - ref.accept_prob).abs().max().item()
        assert diff <= 1e-5, diff
        assert (out.accept_len.cpu().numpy() >= 1).all()
        parity.check_sample(wl, out)
