"""The bounded waits' failure path (needs a GPU).

Kernel A waits, with a time limit, for the logits it stages in shared memory;
a wait that runs out makes the call report SV_REQ_TIMEOUT for every request
(a device fault is the only way the default 2 s limit runs out).  Setting the
limit to 0 makes every such wait give up at once without polling - no fault,
no hang: the kernel still lets its own copies land before it leaves - so the
path can be tested: every request reports the timeout and emits nothing, and
the next call on the same workspace, with the limit restored, is correct."""
import numpy as np
import pytest
import torch

import parity
from token_verification_gb300 import api, synth

pytestmark = pytest.mark.gpu


def _calls(wl_chain, wl_tree):
    d = parity.to_device(wl_chain)
    t = parity.to_device(wl_tree)
    return [
        lambda: api.spec_verify_sample(d["target"], None, d["draft_tokens"], d["uniforms"], 1.0),
        lambda: api.spec_verify_typical(d["target"], d["draft_tokens"], d["uniforms"], 1.0),
        lambda: api.spec_verify_tree_sample(t["target"], t["parent"], t["node_tokens"],
                                            t["uniforms"], 1.0, wl_tree.max_depth),
    ]


def test_zero_wait_limit_reports_timeout_then_recovers():
    wl = synth.make_sample_case(32, 4, 32000, drafts="onehot", seed=70)
    dense = synth.make_sample_case(16, 2, 32000, drafts="dense", seed=71)
    tree = synth.make_tree_case(8, 32000, synth.medusa60_parent(), seed=72)
    tree.uniforms = np.random.default_rng(73).random((8, 61), dtype=np.float32)
    dd = parity.to_device(dense)
    calls = _calls(wl, tree) + [
        lambda: api.spec_verify_sample(dd["target"], dd["draft"], dd["draft_tokens"],
                                       dd["uniforms"], dense.T)]
    default = api.wait_limit_ns()
    assert default == 2_000_000_000
    try:
        api.set_wait_limit_ns(0)
        outs = [c() for c in calls]
        torch.cuda.synchronize()
    finally:
        api.set_wait_limit_ns(default)
    for out in outs:
        assert (out.status.cpu().numpy() == api.REQ_TIMEOUT).all()
        assert (out.accept_len.cpu().numpy() == 0).all()
        assert (out.tokens.cpu().numpy() == -1).all()
    # the same workspaces, the default limit: correct results
    out = calls[0]()
    torch.cuda.synchronize()
    parity.check_sample(wl, out)
    out = calls[3]()
    torch.cuda.synchronize()
    parity.check_sample(dense, out)
    out = calls[2]()
    torch.cuda.synchronize()
    parity.assert_report(parity.compare_tree(tree, out, "sample", 1.0))
