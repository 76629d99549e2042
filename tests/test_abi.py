"""The C-ABI library builds, loads and exports every symbol include/*.h
declares; host-side argument checks return the documented status codes
before any CUDA call (runs without a GPU)."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

from token_verification_gb300 import _native, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", src, flags=re.M):
            if not m.group(0).lstrip().startswith(("#", "typedef", "return")):
                names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _native.lib()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("spec_verify_sample", "spec_verify_greedy", "spec_verify_tree",
              "spec_verify_workspace_size", "spec_verify_workspace_init"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), "libspecverify.so does not export %s" % n
    for n in _native.SYMBOLS:
        assert hasattr(lib, n)
    assert lib.spec_verify_version() == 101


def test_workspace_size(lib):
    assert lib.spec_verify_workspace_size(0, 0, 1) > 0 or lib.spec_verify_workspace_size(0, 0, 1) == 0
    s = lib.spec_verify_workspace_size(256, 5, 152064)
    # at least one 8-byte record per 1024-logit chunk of every row (dense case)
    assert s >= 256 * 11 * 149 * 8 and s % 256 == 0
    assert lib.spec_verify_workspace_size(-1, 5, 10) == 0
    assert lib.spec_verify_workspace_size(4, 32, 10) == 0   # K above the limit
    assert lib.spec_verify_workspace_size(4, 5, 0) == 0


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: every call below fails validation first
NULL = None


def sample(lib, **kw):
    a = dict(target=FAKE, draft=NULL, tokens=FAKE, uniforms=FAKE, T=1.0, out_tokens=FAKE,
             out_len=FAKE, dtype=1, B=4, K=3, V=100, lens=NULL, cu=NULL, packed=NULL, bid=NULL,
             prob=NULL, status=NULL, ws=FAKE, ws_bytes=0, stream=NULL)
    a.update(kw)
    return lib.spec_verify_sample(a["target"], a["draft"], a["tokens"], a["uniforms"],
                                  ctypes.c_float(a["T"]), a["out_tokens"], a["out_len"], a["dtype"],
                                  a["B"], a["K"], a["V"], a["lens"], a["cu"], a["packed"], a["bid"],
                                  a["prob"], a["status"], a["ws"], a["ws_bytes"], a["stream"])


def test_host_validation_codes(lib):
    assert sample(lib, T=-1.0) == 4
    assert sample(lib, T=float("nan")) == 4
    assert sample(lib, T=float("inf")) == 4
    assert sample(lib, dtype=5) == 3
    assert sample(lib, K=32) == 2
    assert sample(lib, V=0) == 2
    assert sample(lib, B=-3) == 2
    assert sample(lib, target=NULL) == 1
    assert sample(lib, tokens=NULL) == 1
    assert sample(lib, uniforms=NULL) == 1
    assert sample(lib, out_len=NULL) == 1
    assert sample(lib, ws=NULL) == 6
    assert sample(lib, ws=ctypes.c_void_p(0x10010)) == 6        # not 256-byte aligned
    assert sample(lib, ws_bytes=100) == 6                        # too small
    need = lib.spec_verify_workspace_size(4, 3, 100)
    assert sample(lib, ws_bytes=need - 1, draft=FAKE) == 6       # dense needs the full size
    g = lib.spec_verify_greedy(NULL, FAKE, FAKE, FAKE, 1, 4, 3, 100, NULL, NULL, NULL, NULL,
                               NULL, FAKE, 0, NULL)
    assert g == 1


def tree(lib, N, max_depth, stride=0, **kw):
    """The greedy tree call with fake device pointers (host checks only: the
    parent array now lives in device memory and is checked there)."""
    return lib.spec_verify_tree(kw.get("target", FAKE), kw.get("parent", FAKE), stride, FAKE,
                                FAKE, FAKE, 1, 2, N, 64, max_depth, NULL, NULL, NULL)


def test_tree_host_validation(lib):
    assert tree(lib, 3, 4, stride=1) == 5            # a parent stride neither 0 nor N
    assert tree(lib, 3, 4, stride=-3) == 5
    assert tree(lib, 257, 2) == 2                    # too many nodes
    assert tree(lib, 3, -1) == 2                     # negative max_depth
    assert tree(lib, 2, 2, target=NULL) == 1
    assert tree(lib, 2, 2, parent=NULL) == 1
    ts = lib.spec_verify_tree_sample(FAKE, FAKE, 0, FAKE, FAKE, ctypes.c_float(-1.0), FAKE, FAKE,
                                     1, 2, 3, 64, 4, NULL, NULL, FAKE, 0, NULL)
    assert ts == 4                                   # negative temperature
    ts = lib.spec_verify_tree_sample(FAKE, FAKE, 0, FAKE, NULL, ctypes.c_float(1.0), FAKE, FAKE,
                                     1, 2, 3, 64, 4, NULL, NULL, FAKE, 0, NULL)
    assert ts == 1                                   # uniforms missing
    ts = lib.spec_verify_tree_sample(FAKE, FAKE, 0, FAKE, FAKE, ctypes.c_float(1.0), FAKE, FAKE,
                                     1, 2, 3, 64, 4, NULL, NULL, FAKE, 0, NULL)
    assert ts == 6                                   # workspace too small


def test_wait_limit_setting(lib):
    """The process-wide wait limit round-trips (no GPU involved)."""
    old = lib.spec_verify_wait_limit_ns()
    assert old == 2_000_000_000
    try:
        assert lib.spec_verify_set_wait_limit_ns(12345) == 0
        assert lib.spec_verify_wait_limit_ns() == 12345
    finally:
        lib.spec_verify_set_wait_limit_ns(old)
    assert lib.spec_verify_wait_limit_ns() == old


def test_status_strings(lib):
    for code in range(8):
        assert lib.spec_verify_status_string(code)
