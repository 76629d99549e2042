"""fp64 CPU oracle for the speculative-decoding verification step.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA product
path never imports it, shares no code with it and never falls back to it.

The arithmetic lives in ``spec_oracle.c`` (plain serial double-precision
loops, one request at a time; see its header for the pages each step
follows).  This module only builds that file with the system C compiler,
marshals numpy arrays into it and, for speed on large inputs, runs disjoint
request ranges on a thread pool (ctypes releases the GIL during a call).

Logit arrays are numpy ``float32`` (fp32 logits) or ``uint16`` holding raw
bfloat16 bit patterns.  Uniform arrays are widened to float64 exactly.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_oracle.c")
_LIB = os.path.join(_HERE, "libspecoracle.so")
_lock = threading.Lock()
_lib = None

BAD_TOKEN = 1
BAD_LOGITS = 2
BAD_DRAFT_LEN = 4
BAD_TREE = 16
FLAG_ACCEPT = 1
FLAG_CDF = 2
FLAG_CUT = 4
FLAG_TOL = 1e-5


def build(force: bool = False) -> str:
    """Compile spec_oracle.c into libspecoracle.so next to it (if stale)."""
    with _lock:
        if (not force and os.path.exists(_LIB)
                and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
            return _LIB
        tmp = _LIB + ".%d.tmp" % os.getpid()
        # ISO C with FP contraction off: the same rounding on x86-64 and AArch64.
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        _lib = configure(ctypes.CDLL(build()))
    return _lib


def configure(lib):
    """Declare the C signatures on a loaded copy of the oracle library."""
    P = ctypes.c_void_p
    I = ctypes.c_int
    D = ctypes.c_double
    lib.sv_oracle_tempered_softmax.argtypes = [P, I, D, P]
    lib.sv_oracle_tempered_softmax.restype = None
    lib.sv_oracle_argmax.argtypes = [P, I]
    lib.sv_oracle_argmax.restype = I
    lib.sv_oracle_inverse_cdf.argtypes = [P, I, D, P]
    lib.sv_oracle_inverse_cdf.restype = I
    lib.sv_oracle_greedy.argtypes = [P, I, P, P, I, I, I, I, I, P, P, P, P]
    lib.sv_oracle_greedy.restype = I
    lib.sv_oracle_sample.argtypes = [P, P, I, P, P, P, D, I, I, I, I, I, P, P, P, P, P, P, P, P,
                                     P, I, D, P, P, P]
    lib.sv_oracle_sample.restype = I
    lib.sv_oracle_tree.argtypes = [P, I, P, I, P, I, I, I, I, I, I, P, P, P, P]
    lib.sv_oracle_tree.restype = I
    lib.sv_oracle_compact.argtypes = [P, P, I, I, P, P, P]
    lib.sv_oracle_compact.restype = None
    lib.sv_oracle_typical.argtypes = [P, I, P, P, P, D, D, D, I, I, I, I, I, P, P, P, P, P, P, P,
                                      P, P]
    lib.sv_oracle_typical.restype = I
    lib.sv_oracle_tree_typical.argtypes = [P, I, P, I, P, P, D, D, D, I, I, I, I, I, I, P, P, P,
                                           P, P, P, P, P, P, P]
    lib.sv_oracle_tree_sample.argtypes = [P, I, P, I, P, P, D, I, I, I, I, I, I, P, P, P, P, P,
                                          P, P, P, P, P, P]
    lib.sv_oracle_tree_sample.restype = I
    lib.sv_oracle_tree_typical.restype = I
    lib.sv_oracle_ngram.argtypes = [P, P, I, I, I, I, I, P, P, P, P, P]
    lib.sv_oracle_ngram.restype = I
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _logits(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, 0
    if a.dtype == np.uint16:
        return a, 1
    raise TypeError("oracle logits must be float32 or uint16 (bfloat16 bits), got %s" % a.dtype)


def _mask(token_mask, B, K1, V):
    """Grammar masks as contiguous uint32 [B, K+1, ceil(V/32)] (or None)."""
    if token_mask is None:
        return None
    m = np.ascontiguousarray(token_mask)
    if m.dtype not in (np.int32, np.uint32) or m.shape != (B, K1, (V + 31) // 32):
        raise ValueError("token_mask must be int32/uint32 [B, K+1, ceil(V/32)]")
    return m.view(np.uint32)


def _ranges(B, threads):
    threads = max(1, min(int(threads), B)) if B > 0 else 1
    edges = np.linspace(0, B, threads + 1).astype(int)
    return [(int(edges[i]), int(edges[i + 1])) for i in range(threads)]


def _run(fn, B, threads, b_range):
    lo, hi = (0, B) if b_range is None else b_range
    parts = [(lo + a, lo + b) for a, b in _ranges(hi - lo, threads)]
    if len(parts) == 1:
        rc = fn(*parts[0])
        if rc != 0:
            raise ValueError("oracle rejected its arguments (code %d)" % rc)
        return
    with ThreadPoolExecutor(len(parts)) as ex:
        for rc in ex.map(lambda ab: fn(*ab), parts):
            if rc != 0:
                raise ValueError("oracle rejected its arguments (code %d)" % rc)


# ---------------------------------------------------------------------------
# single steps (exposed so that the tests can pin them against library code)
# ---------------------------------------------------------------------------

def tempered_softmax(logits, temperature):
    l = np.ascontiguousarray(logits, dtype=np.float64)
    out = np.empty_like(l)
    _load().sv_oracle_tempered_softmax(_ptr(l), l.size, float(temperature), _ptr(out))
    return out


def argmax(logits):
    l = np.ascontiguousarray(logits, dtype=np.float64)
    return int(_load().sv_oracle_argmax(_ptr(l), l.size))


def inverse_cdf(weights, u):
    w = np.ascontiguousarray(weights, dtype=np.float64)
    m = np.zeros(1, dtype=np.float64)
    t = _load().sv_oracle_inverse_cdf(_ptr(w), w.size, float(u), _ptr(m))
    return int(t), float(m[0])


# ---------------------------------------------------------------------------
# batched verification
# ---------------------------------------------------------------------------

def sample(target, draft, draft_tokens, uniforms, temperature, *, draft_lens=None,
           threads=1, b_range=None, probe_tokens=None, token_mask=None, top_k=0, top_p=1.0,
           flip=None, cut_logits=None):
    """Rejection-sampling verify (temperature 0 = greedy rule).

    target [B, K+1, V], draft [B, K, V] or None (one-hot drafts),
    draft_tokens [B, K] int32, uniforms [B, K+1] (float32 or float64),
    draft_lens [B] or None.  Requests outside ``b_range`` keep -1 / 0.
    token_mask [B, K+1, ceil(V/32)] int32 / uint32 or None: grammar masks
    (bit j % 32 of word j // 32 set = token j allowed at that position).
    top_k (0 = off) and top_p (1.0 = off) filter every sampled distribution,
    target and dense draft alike; flags gain FLAG_CUT where a top-p cut is
    within FLAG_TOL of moving.
    flip [B, K] (bool / uint8) or None: invert the outcome of the marked
    acceptance tests (to follow the other branch of a flagged test).
    cut_logits [B, R] or None (R = K+1, plus K with draft logits: target rows
    then draft rows; NaN = the rule's own cut): forced top-p cuts; the result
    gains cut_margin [B, R] (0 = the rule's own cut, d > 0 = a different cut
    at distance d <= FLAG_TOL from the rule, NaN = not admissible, -1 = row
    not reached).
    Returns a dict of numpy arrays: tokens, accept_len, accept_prob, flags,
    margins, status (and probe [B, 2] when probe_tokens [B] is given: the
    normalised CDF step of that token in the request's final draw).
    """
    target, dt = _logits(target)
    B, K1, V = target.shape
    K = K1 - 1
    if draft is not None:
        draft, dt2 = _logits(draft)
        if dt2 != dt or draft.shape != (B, K, V):
            raise ValueError("draft logits must match target dtype and be [B, K, V]")
    toks = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, K)
    u = np.ascontiguousarray(uniforms, dtype=np.float64).reshape(B, K + 1)
    lens = None if draft_lens is None else np.ascontiguousarray(draft_lens, dtype=np.int32)
    mask = _mask(token_mask, B, K + 1, V)
    out = dict(tokens=np.full((B, K + 1), -1, np.int32), accept_len=np.zeros(B, np.int32),
               accept_prob=np.full((B, K), -1.0), flags=np.zeros((B, K + 1), np.int32),
               margins=np.full((B, K + 1), np.inf), status=np.zeros(B, np.int32))
    probes = None
    if probe_tokens is not None:
        probes = np.ascontiguousarray(probe_tokens, dtype=np.int32).reshape(B)
        out["probe"] = np.full((B, 2), np.nan)
    fl = None if flip is None else np.ascontiguousarray(flip, dtype=np.uint8).reshape(B, K)
    cuts = None
    if cut_logits is not None:
        R = K + 1 + (K if draft is not None else 0)
        cuts = np.ascontiguousarray(cut_logits, dtype=np.float64).reshape(B, R)
        out["cut_margin"] = np.full((B, R), -1.0)
    lib = _load()

    def fn(lo, hi):
        return lib.sv_oracle_sample(
            _ptr(target), _ptr(draft), dt, _ptr(toks), _ptr(lens), _ptr(u),
            float(temperature), B, K, V, lo, hi, _ptr(out["tokens"]), _ptr(out["accept_len"]),
            _ptr(out["accept_prob"]), _ptr(out["flags"]), _ptr(out["margins"]),
            _ptr(out["status"]), _ptr(probes), _ptr(out.get("probe")), _ptr(mask), int(top_k),
            float(top_p), _ptr(fl), _ptr(cuts), _ptr(out.get("cut_margin")))

    _run(fn, B, threads, b_range)
    return out


def greedy(target, draft_tokens, *, draft_lens=None, threads=1, b_range=None, token_mask=None):
    """Greedy verify: tokens [B, K+1], accept_len [B], status [B]
    (token_mask as for ``sample``)."""
    target, dt = _logits(target)
    B, K1, V = target.shape
    K = K1 - 1
    mask = _mask(token_mask, B, K1, V)
    toks = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, K)
    lens = None if draft_lens is None else np.ascontiguousarray(draft_lens, dtype=np.int32)
    out = dict(tokens=np.full((B, K + 1), -1, np.int32), accept_len=np.zeros(B, np.int32),
               status=np.zeros(B, np.int32))
    lib = _load()

    def fn(lo, hi):
        return lib.sv_oracle_greedy(_ptr(target), dt, _ptr(toks), _ptr(lens), B, K, V, lo, hi,
                                    _ptr(out["tokens"]), _ptr(out["accept_len"]),
                                    _ptr(out["status"]), _ptr(mask))

    _run(fn, B, threads, b_range)
    return out


def _parents(parent, B, N):
    """A shared parent array [N] (stride 0) or one per request [B, N] (stride N)."""
    par = np.ascontiguousarray(parent, dtype=np.int32)
    if par.shape == (N,):
        return par, 0
    if par.shape == (B, N):
        return par, N
    raise ValueError("parent must be [N] or [B, N] (N = %d, B = %d), got %s" % (N, B, par.shape))


def tree(target, parent, node_tokens, max_depth, *, threads=1, b_range=None):
    """Greedy tree verify: tokens / path [B, max_depth+1], accept_len, status.
    parent: [N] shared by every request, or [B, N] (one tree per request)."""
    target, dt = _logits(target)
    B, N1, V = target.shape
    N = N1 - 1
    par, stride = _parents(parent, B, N)
    nt = np.ascontiguousarray(node_tokens, dtype=np.int32).reshape(B, N)
    W = max_depth + 1
    out = dict(tokens=np.full((B, W), -1, np.int32), accept_len=np.zeros(B, np.int32),
               path=np.full((B, W), -1, np.int32), status=np.zeros(B, np.int32))
    lib = _load()

    def fn(lo, hi):
        return lib.sv_oracle_tree(_ptr(target), dt, _ptr(par), stride, _ptr(nt), B, N, V,
                                  int(max_depth), lo, hi, _ptr(out["tokens"]),
                                  _ptr(out["accept_len"]), _ptr(out["path"]), _ptr(out["status"]))

    _run(fn, B, threads, b_range)
    return out


def tree_sample(target, parent, node_tokens, uniforms, temperature, max_depth, *, threads=1,
                b_range=None, flip=None, probe_tokens=None):
    """Lossless tree verification by rejection sampling over deterministic
    candidates.  parent [N] or [B, N]; uniforms [B, N+1] (column n drives the
    test of node n, column 0 the final draw).  Returns tokens / path
    [B, max_depth+1], accept_len, accept_prob [B, N+1] (theta of each tested
    node, -1 elsewhere), node_flags [B, N+1] (FLAG_ACCEPT per flagged test),
    flags [B] (FLAG_CDF for the draw), margins [B], status (and probe [B, 2]
    with probe_tokens [B]).  flip [B, N+1] inverts the marked node tests."""
    target, dt = _logits(target)
    B, N1, V = target.shape
    N = N1 - 1
    par, stride = _parents(parent, B, N)
    nt = np.ascontiguousarray(node_tokens, dtype=np.int32).reshape(B, N)
    u = np.ascontiguousarray(uniforms, dtype=np.float64).reshape(B, N + 1)
    fl = None if flip is None else np.ascontiguousarray(flip, dtype=np.uint8).reshape(B, N + 1)
    W = max_depth + 1
    out = dict(tokens=np.full((B, W), -1, np.int32), accept_len=np.zeros(B, np.int32),
               path=np.full((B, W), -1, np.int32), accept_prob=np.full((B, N + 1), -1.0),
               node_flags=np.zeros((B, N + 1), np.int32), flags=np.zeros(B, np.int32),
               margins=np.full(B, np.inf), status=np.zeros(B, np.int32))
    probes = None
    if probe_tokens is not None:
        probes = np.ascontiguousarray(probe_tokens, dtype=np.int32).reshape(B)
        out["probe"] = np.full((B, 2), np.nan)
    lib = _load()

    def fn(lo, hi):
        return lib.sv_oracle_tree_sample(
            _ptr(target), dt, _ptr(par), stride, _ptr(nt), _ptr(u), float(temperature), B, N, V,
            int(max_depth), lo, hi, _ptr(fl), _ptr(out["tokens"]), _ptr(out["accept_len"]),
            _ptr(out["path"]), _ptr(out["accept_prob"]), _ptr(out["node_flags"]),
            _ptr(out["flags"]), _ptr(out["margins"]), _ptr(out["status"]), _ptr(probes),
            _ptr(out.get("probe")))

    _run(fn, B, threads, b_range)
    return out


def typical(target, draft_tokens, uniforms, temperature, eps, delta, *, draft_lens=None,
            threads=1, b_range=None, flip=None, probe_tokens=None):
    """Typical acceptance: accept x_i while p_i(x_i) > min(eps, delta *
    exp(-H(p_i))); the emitted token at the first failure (or the bonus
    position) is drawn from p_n with uniforms[:, K].  Returns tokens,
    accept_len, accept_prob (p_i(x_i) at tested positions), flags, margins
    [B] (the draw's distance to its CDF step's nearer edge), status (and
    probe [B, 2] with probe_tokens [B]).  flip [B, K] inverts the marked
    tests."""
    target, dt = _logits(target)
    B, K1, V = target.shape
    K = K1 - 1
    toks = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, K)
    u = np.ascontiguousarray(uniforms, dtype=np.float64).reshape(B, K + 1)
    lens = None if draft_lens is None else np.ascontiguousarray(draft_lens, dtype=np.int32)
    out = dict(tokens=np.full((B, K + 1), -1, np.int32), accept_len=np.zeros(B, np.int32),
               accept_prob=np.full((B, K), -1.0), flags=np.zeros((B, K + 1), np.int32),
               margins=np.full(B, np.inf), status=np.zeros(B, np.int32))
    fl = None if flip is None else np.ascontiguousarray(flip, dtype=np.uint8).reshape(B, K)
    probes = None
    if probe_tokens is not None:
        probes = np.ascontiguousarray(probe_tokens, dtype=np.int32).reshape(B)
        out["probe"] = np.full((B, 2), np.nan)
    lib = _load()

    def fn(lo, hi):
        return lib.sv_oracle_typical(_ptr(target), dt, _ptr(toks), _ptr(lens), _ptr(u),
                                     float(temperature), float(eps), float(delta), B, K, V, lo, hi,
                                     _ptr(out["tokens"]), _ptr(out["accept_len"]),
                                     _ptr(out["accept_prob"]), _ptr(out["flags"]),
                                     _ptr(out["status"]), _ptr(fl), _ptr(out["margins"]),
                                     _ptr(probes), _ptr(out.get("probe")))

    _run(fn, B, threads, b_range)
    return out


def tree_typical(target, parent, node_tokens, uniforms, temperature, eps, delta, max_depth, *,
                 threads=1, b_range=None, flip=None, probe_tokens=None):
    """Typical acceptance over a candidate tree: tokens / path [B, max_depth+1],
    accept_len, flags [B], node_flags [B, N+1] (FLAG_ACCEPT per flagged node
    test), margins [B], status (and probe [B, 2] with probe_tokens [B]).
    parent [N] or [B, N]; uniforms [B] drive the final draw; flip [B, N+1]
    inverts the marked node tests."""
    target, dt = _logits(target)
    B, N1, V = target.shape
    N = N1 - 1
    par, stride = _parents(parent, B, N)
    nt = np.ascontiguousarray(node_tokens, dtype=np.int32).reshape(B, N)
    u = np.ascontiguousarray(uniforms, dtype=np.float64).reshape(B)
    fl = None if flip is None else np.ascontiguousarray(flip, dtype=np.uint8).reshape(B, N + 1)
    W = max_depth + 1
    out = dict(tokens=np.full((B, W), -1, np.int32), accept_len=np.zeros(B, np.int32),
               path=np.full((B, W), -1, np.int32), flags=np.zeros(B, np.int32),
               node_flags=np.zeros((B, N + 1), np.int32), margins=np.full(B, np.inf),
               status=np.zeros(B, np.int32))
    probes = None
    if probe_tokens is not None:
        probes = np.ascontiguousarray(probe_tokens, dtype=np.int32).reshape(B)
        out["probe"] = np.full((B, 2), np.nan)
    lib = _load()

    def fn(lo, hi):
        return lib.sv_oracle_tree_typical(_ptr(target), dt, _ptr(par), stride, _ptr(nt), _ptr(u),
                                          float(temperature), float(eps), float(delta), B, N, V,
                                          int(max_depth), lo, hi, _ptr(out["tokens"]),
                                          _ptr(out["accept_len"]), _ptr(out["path"]),
                                          _ptr(out["flags"]), _ptr(out["status"]), _ptr(fl),
                                          _ptr(out["node_flags"]), _ptr(out["margins"]),
                                          _ptr(probes), _ptr(out.get("probe")))

    _run(fn, B, threads, b_range)
    return out


def compact(tokens, accept_len):
    """Padding-free layout: cu [B+1], packed [B*W], batch_id [B*W]."""
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    a = np.ascontiguousarray(accept_len, dtype=np.int32)
    B, W = t.shape
    cu = np.zeros(B + 1, np.int32)
    packed = np.empty(B * W, np.int32)
    bid = np.empty(B * W, np.int32)
    _load().sv_oracle_compact(_ptr(t), _ptr(a), B, W, _ptr(cu), _ptr(packed), _ptr(bid))
    return cu, packed, bid



def ngram(tokens, lens, n_min, n_max, K):
    """Prompt-lookup proposer: drafts [B, K] (-1 padded), draft_lens [B],
    match [B] (start of the matched n-gram or -1), ngram [B] (its n or 0),
    status [B] (BAD_DRAFT_LEN for a context length outside [0, L])."""
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    B, L = t.shape
    ln = np.ascontiguousarray(lens, dtype=np.int32).reshape(B)
    out = dict(drafts=np.full((B, K), -1, np.int32), draft_lens=np.zeros(B, np.int32),
               match=np.full(B, -1, np.int32), ngram=np.zeros(B, np.int32),
               status=np.zeros(B, np.int32))
    rc = _load().sv_oracle_ngram(_ptr(t), _ptr(ln), B, L, int(n_min), int(n_max), int(K),
                                 _ptr(out["drafts"]), _ptr(out["draft_lens"]), _ptr(out["match"]),
                                 _ptr(out["ngram"]), _ptr(out["status"]))
    if rc != 0:
        raise ValueError("oracle rejected its arguments (code %d)" % rc)
    return out
