"""Python binding of the C ABI: argument marshalling only.

Every step of the verification runs in the CUDA kernels of libspecverify;
PyTorch provides device memory and the current stream.  Function names and
argument order follow include/spec_verify.h.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from . import _native

SV_F32 = 0
SV_BF16 = 1
REQ_BAD_TOKEN = 1
REQ_BAD_LOGITS = 2
REQ_BAD_DRAFT_LEN = 4
REQ_TIMEOUT = 8
REQ_BAD_TREE = 16
MAX_K = 31


class VerifyError(RuntimeError):
    def __init__(self, code):
        msg = _native.lib().spec_verify_status_string(int(code)).decode()
        super().__init__("spec_verify failed (%d): %s" % (code, msg))
        self.code = int(code)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_F32
    raise TypeError("logits must be torch.bfloat16 or torch.float32, got %s" % t.dtype)


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(t: torch.Tensor, name, device, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.device != device:
        raise ValueError("%s must be on %s (got %s)" % (name, device, t.device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s (got %s)" % (name, dtype, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s (got %s)" % (name, tuple(shape), tuple(t.shape)))


# ---------------------------------------------------------------------------
# workspaces: one per (device, stream), grown on demand, zero-filled once
# ---------------------------------------------------------------------------

_workspaces = {}


def workspace(B: int, K: int, V: int, device: torch.device, *, need: Optional[int] = None):
    """The (device, stream)'s workspace, grown to the bytes a (B, K, V) call
    needs (or to ``need`` bytes when given)."""
    lib = _native.lib()
    if need is None:
        need = int(lib.spec_verify_workspace_size(B, K, V))
    if need == 0 and B > 0:
        raise ValueError("unsupported shape B=%d K=%d V=%d" % (B, K, V))
    stream = torch.cuda.current_stream(device)
    key = (device.index, stream.cuda_stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        rc = lib.spec_verify_workspace_init(_p(ws), ws.numel(), _stream(device))
        if rc:
            raise VerifyError(rc)
        _workspaces[key] = ws
    return ws


@dataclass
class VerifyOutputs:
    tokens: torch.Tensor           # [B, K+1] int32
    accept_len: torch.Tensor       # [B] int32
    cu_accept: Optional[torch.Tensor] = None   # [B+1]
    packed: Optional[torch.Tensor] = None      # [B*(K+1)]
    batch_id: Optional[torch.Tensor] = None    # [B*(K+1)]
    accept_prob: Optional[torch.Tensor] = None  # [B, K] fp32
    status: Optional[torch.Tensor] = None      # [B]
    cut: Optional[torch.Tensor] = None         # [B, R] fp32 (filtered calls)


def alloc_outputs(B, K, device, *, packed=True, accept_prob=True, status=True):
    i32 = dict(dtype=torch.int32, device=device)
    return VerifyOutputs(
        tokens=torch.empty((B, K + 1), **i32), accept_len=torch.empty((B,), **i32),
        cu_accept=torch.empty((B + 1,), **i32) if packed else None,
        packed=torch.empty((B * (K + 1),), **i32) if packed else None,
        batch_id=torch.empty((B * (K + 1),), **i32) if packed else None,
        accept_prob=torch.empty((B, K), dtype=torch.float32, device=device) if accept_prob else None,
        status=torch.empty((B,), **i32) if status else None)


def _validate_batch(target_logits, draft_tokens, draft_lens):
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, K+1, V]")
    B, K1, V = target_logits.shape
    K = K1 - 1
    device = target_logits.device
    if device.type != "cuda":
        raise ValueError("target_logits must be a CUDA tensor")
    _check(target_logits, "target_logits", device)
    if K > 0 or draft_tokens is not None:
        _check(draft_tokens, "draft_tokens", device, torch.int32, (B, K))
    if draft_lens is not None:
        _check(draft_lens, "draft_lens", device, torch.int32, (B,))
    return B, K, V, device


def _check_mask(token_mask, B, K, V, device):
    if token_mask is not None:
        _check(token_mask, "token_mask", device, torch.int32, (B, K + 1, (V + 31) // 32))


def spec_verify_sample(target_logits, draft_logits, draft_tokens, uniforms, temperature,
                       out: Optional[VerifyOutputs] = None, *, draft_lens=None,
                       packed=True, accept_prob=True, status=True,
                       token_mask=None, top_k=0, top_p=1.0, cut=False) -> VerifyOutputs:
    """Rejection-sampling verification of one batch (see spec_verify.h).

    target_logits [B, K+1, V] bf16/fp32 CUDA; draft_logits [B, K, V] same
    dtype or None (one-hot drafts); draft_tokens [B, K] int32; uniforms
    [B, K+1] fp32; temperature >= 0 (0 = greedy rule); token_mask
    [B, K+1, ceil(V/32)] int32 grammar masks or None (bit j % 32 of word
    j // 32 set = token j allowed at that position); top_k (0 = off) and
    top_p (1.0 = off) filter every sampled distribution; cut=True (filtered
    calls) also returns out.cut [B, R], each row's lowest kept logit (R =
    K+1 target rows, then K draft rows with draft logits)."""
    B, K, V, device = _validate_batch(target_logits, draft_tokens, draft_lens)
    if draft_logits is not None:
        _check(draft_logits, "draft_logits", device, target_logits.dtype, (B, K, V))
    _check(uniforms, "uniforms", device, torch.float32, (B, K + 1))
    _check_mask(token_mask, B, K, V, device)
    if out is None:
        out = alloc_outputs(B, K, device, packed=packed, accept_prob=accept_prob, status=status)
    filtered = top_k != 0 or top_p != 1.0
    if filtered and cut and out.cut is None:
        R = K + 1 + (K if draft_logits is not None else 0)
        out.cut = torch.empty((B, R), dtype=torch.float32, device=device)
    ws = workspace(B, K, V, device)
    lib = _native.lib()
    head = (_p(target_logits), _p(draft_logits), _p(draft_tokens), _p(uniforms),
            ctypes.c_float(float(temperature)))
    mid = (_p(out.tokens), _p(out.accept_len), _dtype_code(target_logits), B, K, V,
           _p(draft_lens), _p(out.cu_accept), _p(out.packed), _p(out.batch_id),
           _p(out.accept_prob))
    end = (_p(out.status), _p(ws), ws.numel(), _stream(device))
    tail = mid + end
    if filtered:
        rc = lib.spec_verify_sample_filtered(*head, int(top_k), ctypes.c_float(float(top_p)),
                                             _p(token_mask), *mid,
                                             _p(out.cut if cut else None), *end)
    elif token_mask is None:
        rc = lib.spec_verify_sample(*head, *tail)
    else:
        rc = lib.spec_verify_sample_masked(*head, _p(token_mask), *tail)
    if rc:
        raise VerifyError(rc)
    return out


def spec_verify_greedy(target_logits, draft_tokens, out: Optional[VerifyOutputs] = None, *,
                       draft_lens=None, packed=True, status=True,
                       token_mask=None) -> VerifyOutputs:
    """Greedy verification: accept while the draft equals the target argmax
    (over the tokens token_mask allows, when given)."""
    B, K, V, device = _validate_batch(target_logits, draft_tokens, draft_lens)
    _check_mask(token_mask, B, K, V, device)
    if out is None:
        out = alloc_outputs(B, K, device, packed=packed, accept_prob=False, status=status)
    ws = workspace(B, K, V, device)
    lib = _native.lib()
    tail = (_p(out.tokens), _p(out.accept_len), _dtype_code(target_logits), B, K, V,
            _p(draft_lens), _p(out.cu_accept), _p(out.packed), _p(out.batch_id), _p(out.status),
            _p(ws), ws.numel(), _stream(device))
    if token_mask is None:
        rc = lib.spec_verify_greedy(_p(target_logits), _p(draft_tokens), *tail)
    else:
        rc = lib.spec_verify_greedy_masked(_p(target_logits), _p(draft_tokens), _p(token_mask),
                                           *tail)
    if rc:
        raise VerifyError(rc)
    return out


@dataclass
class TreeOutputs:
    tokens: torch.Tensor      # [B, max_depth+1]
    accept_len: torch.Tensor  # [B]
    path: Optional[torch.Tensor] = None
    status: Optional[torch.Tensor] = None


def tree_depth(parent) -> int:
    """Depth of a host-side parent array (parent of node n at index n-1)."""
    d = [0]
    for n, p in enumerate(np.asarray(parent, dtype=np.int64).reshape(-1), start=1):
        if p < 0 or p >= n:
            raise ValueError("parent of node %d must be an earlier node (got %d)" % (n, p))
        d.append(d[p] + 1)
    return max(d)


def _tree_args(target_logits, tree_parent, tree_tokens, max_depth):
    """(B, N, V, device, parent tensor, parent stride, max_depth).  tree_parent:
    a CUDA int32 tensor [N] (one tree) or [B, N] (a tree per request) - then
    max_depth must be given - or a host array [N] / [B, N], copied to the
    device, whose depth is the default max_depth."""
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, N+1, V]")
    B, N1, V = target_logits.shape
    N = N1 - 1
    device = target_logits.device
    _check(target_logits, "target_logits", device)
    if not (isinstance(tree_parent, torch.Tensor) and tree_parent.device == device):
        host = np.ascontiguousarray(np.asarray(tree_parent, dtype=np.int32))
        if max_depth is None:
            max_depth = max(tree_depth(r) for r in host.reshape(-1, N)) if N else 0
        tree_parent = torch.from_numpy(host).to(device)
    if max_depth is None:
        raise ValueError("max_depth is required with a device-side tree_parent")
    if tuple(tree_parent.shape) == (N,):
        stride = 0
    elif tuple(tree_parent.shape) == (B, N):
        stride = N
    else:
        raise ValueError("tree_parent must be [N] or [B, N] (N = %d)" % N)
    _check(tree_parent, "tree_parent", device, torch.int32)
    _check(tree_tokens, "tree_tokens", device, torch.int32, (B, N))
    return B, N, V, device, tree_parent, stride, int(max_depth)


def _tree_outputs(B, D1, device, path, status):
    i32 = dict(dtype=torch.int32, device=device)
    return TreeOutputs(tokens=torch.empty((B, D1), **i32), accept_len=torch.empty((B,), **i32),
                       path=torch.empty((B, D1), **i32) if path else None,
                       status=torch.empty((B,), **i32) if status else None)


def spec_verify_tree(target_logits, tree_parent, tree_tokens, max_depth=None,
                     out: Optional[TreeOutputs] = None, *, path=True, status=True) -> TreeOutputs:
    """Greedy tree verification.  tree_parent [N] or [B, N] (parent of node n
    at index n-1; device tensor, or host array copied to the device);
    tree_tokens [B, N] int32 CUDA."""
    B, N, V, device, par, stride, max_depth = _tree_args(target_logits, tree_parent, tree_tokens,
                                                         max_depth)
    if out is None:
        out = _tree_outputs(B, max_depth + 1, device, path, status)
    rc = _native.lib().spec_verify_tree(
        _p(target_logits), _p(par), stride, _p(tree_tokens), _p(out.tokens), _p(out.accept_len),
        _dtype_code(target_logits), B, N, V, max_depth, _p(out.path), _p(out.status),
        _stream(device))
    if rc:
        raise VerifyError(rc)
    return out


def spec_verify_tree_sample(target_logits, tree_parent, tree_tokens, uniforms, temperature,
                            max_depth=None, out: Optional[TreeOutputs] = None, *, path=True,
                            status=True) -> TreeOutputs:
    """Lossless tree verification by rejection sampling (see spec_verify.h):
    tree_parent as for spec_verify_tree, tree_tokens [B, N] int32, uniforms
    [B, N+1] fp32 (column n: node n's test, column 0: the final draw);
    temperature 0 runs the greedy walk."""
    B, N, V, device, par, stride, max_depth = _tree_args(target_logits, tree_parent, tree_tokens,
                                                         max_depth)
    _check(uniforms, "uniforms", device, torch.float32, (B, N + 1))
    if out is None:
        out = _tree_outputs(B, max_depth + 1, device, path, status)
    lib = _native.lib()
    ws = workspace(B, N, V, device, need=int(lib.spec_verify_tree_workspace_size(B, N, V)))
    rc = lib.spec_verify_tree_sample(
        _p(target_logits), _p(par), stride, _p(tree_tokens), _p(uniforms),
        ctypes.c_float(float(temperature)), _p(out.tokens), _p(out.accept_len),
        _dtype_code(target_logits), B, N, V, max_depth, _p(out.path), _p(out.status), _p(ws),
        ws.numel(), _stream(device))
    if rc:
        raise VerifyError(rc)
    return out


def spec_verify_typical(target_logits, draft_tokens, uniforms, temperature, eps=0.09, delta=0.3,
                        out: Optional[VerifyOutputs] = None, *, draft_lens=None, packed=True,
                        accept_prob=True, status=True) -> VerifyOutputs:
    """Typical acceptance (see spec_verify.h): x_i passes while p_i(x_i) >
    min(eps, delta * exp(-H(p_i))); the token after the accepted ones is
    drawn from the target distribution there with uniforms[:, K]."""
    B, K, V, device = _validate_batch(target_logits, draft_tokens, draft_lens)
    _check(uniforms, "uniforms", device, torch.float32, (B, K + 1))
    if out is None:
        out = alloc_outputs(B, K, device, packed=packed, accept_prob=accept_prob, status=status)
    ws = workspace(B, K, V, device)
    rc = _native.lib().spec_verify_typical(
        _p(target_logits), _p(draft_tokens), _p(uniforms), ctypes.c_float(float(temperature)),
        ctypes.c_float(float(eps)), ctypes.c_float(float(delta)), _p(out.tokens),
        _p(out.accept_len), _dtype_code(target_logits), B, K, V, _p(draft_lens), _p(out.cu_accept),
        _p(out.packed), _p(out.batch_id), _p(out.accept_prob), _p(out.status), _p(ws), ws.numel(),
        _stream(device))
    if rc:
        raise VerifyError(rc)
    return out


def spec_verify_tree_typical(target_logits, tree_parent, tree_tokens, uniforms, temperature,
                             eps=0.09, delta=0.3, max_depth=None,
                             out: Optional[TreeOutputs] = None, *, path=True,
                             status=True) -> TreeOutputs:
    """Typical acceptance over a candidate tree: tree_parent as for
    spec_verify_tree, tree_tokens [B, N] int32, uniforms [B] fp32 for the
    final draw."""
    B, N, V, device, par, stride, max_depth = _tree_args(target_logits, tree_parent, tree_tokens,
                                                         max_depth)
    _check(uniforms, "uniforms", device, torch.float32, (B,))
    if out is None:
        out = _tree_outputs(B, max_depth + 1, device, path, status)
    lib = _native.lib()
    ws = workspace(B, N, V, device, need=int(lib.spec_verify_tree_workspace_size(B, N, V)))
    rc = lib.spec_verify_tree_typical(
        _p(target_logits), _p(par), stride, _p(tree_tokens), _p(uniforms),
        ctypes.c_float(float(temperature)), ctypes.c_float(float(eps)),
        ctypes.c_float(float(delta)), _p(out.tokens), _p(out.accept_len),
        _dtype_code(target_logits), B, N, V, max_depth, _p(out.path), _p(out.status),
        _p(ws), ws.numel(), _stream(device))
    if rc:
        raise VerifyError(rc)
    return out


def set_wait_limit_ns(limit_ns: int) -> None:
    """The longest a kernel waits for staged logits before the call reports
    REQ_TIMEOUT (default 2 s; 0 gives up at once).  Process-wide."""
    _native.lib().spec_verify_set_wait_limit_ns(int(limit_ns))


def wait_limit_ns() -> int:
    return int(_native.lib().spec_verify_wait_limit_ns())


@dataclass
class NgramOutputs:
    drafts: torch.Tensor      # [B, K], -1 after the drafts
    draft_lens: torch.Tensor  # [B]
    match: Optional[torch.Tensor] = None
    status: Optional[torch.Tensor] = None


def spec_ngram_propose(tokens, lens, K=5, n_min=1, n_max=4, out: Optional[NgramOutputs] = None,
                       *, match=True, status=True) -> NgramOutputs:
    """n-gram (prompt-lookup) proposer (see spec_verify.h): tokens [B, L]
    int32 contexts, lens [B] int32.  The drafts feed spec_verify_sample as
    one-hot drafts with draft_lens = out.draft_lens."""
    if tokens.dim() != 2:
        raise ValueError("tokens must be [B, L]")
    B, L = tokens.shape
    device = tokens.device
    if device.type != "cuda":
        raise ValueError("tokens must be a CUDA tensor")
    _check(tokens, "tokens", device, torch.int32)
    _check(lens, "lens", device, torch.int32, (B,))
    if out is None:
        i32 = dict(dtype=torch.int32, device=device)
        out = NgramOutputs(drafts=torch.empty((B, K), **i32), draft_lens=torch.empty((B,), **i32),
                           match=torch.empty((B,), **i32) if match else None,
                           status=torch.empty((B,), **i32) if status else None)
    rc = _native.lib().spec_ngram_propose(_p(tokens), _p(lens), B, L, int(n_min), int(n_max),
                                          int(K), _p(out.drafts), _p(out.draft_lens),
                                          _p(out.match), _p(out.status), _stream(device))
    if rc:
        raise VerifyError(rc)
    return out
