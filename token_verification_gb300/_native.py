"""ctypes declarations of libspecverify.so (include/spec_verify.h).

There is no fallback: if the library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libspecverify.so")

SYMBOLS = (
    "spec_verify_workspace_size", "spec_verify_workspace_init", "spec_verify_sample",
    "spec_verify_greedy", "spec_verify_tree", "spec_verify_status_string",
    "spec_verify_version", "spec_verify_sample_noalloc", "spec_verify_sample_masked",
    "spec_verify_greedy_masked", "spec_ngram_propose", "spec_verify_sample_filtered",
    "spec_verify_typical", "spec_verify_tree_typical", "spec_verify_tree_workspace_size",
    "spec_verify_tree_sample", "spec_verify_set_wait_limit_ns", "spec_verify_wait_limit_ns",
)

_lock = threading.Lock()
_lib = None


def lib():
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libspecverify.so is not built (expected at %s); build it with "
                "token_verification_gb300.build.build()" % LIB_PATH)
        l = ctypes.CDLL(LIB_PATH)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        l.spec_verify_workspace_size.argtypes = [I, I, I]
        l.spec_verify_workspace_size.restype = Z
        l.spec_verify_workspace_init.argtypes = [P, Z, P]
        l.spec_verify_workspace_init.restype = I
        l.spec_verify_sample.argtypes = [P, P, P, P, F, P, P, I, I, I, I, P, P, P, P, P, P, P, Z, P]
        l.spec_verify_sample.restype = I
        l.spec_verify_sample_noalloc.argtypes = [P, P, P, P, F, P, P, I, I, I, I, P, P, P, P, P,
                                                 P, P]
        l.spec_verify_sample_noalloc.restype = I
        l.spec_verify_greedy.argtypes = [P, P, P, P, I, I, I, I, P, P, P, P, P, P, Z, P]
        l.spec_verify_greedy.restype = I
        l.spec_verify_sample_masked.argtypes = [P, P, P, P, F, P, P, P, I, I, I, I, P, P, P, P, P,
                                                P, P, Z, P]
        l.spec_verify_sample_masked.restype = I
        l.spec_verify_greedy_masked.argtypes = [P, P, P, P, P, I, I, I, I, P, P, P, P, P, P, Z, P]
        l.spec_verify_greedy_masked.restype = I
        l.spec_verify_sample_filtered.argtypes = [P, P, P, P, F, I, F, P, P, P, I, I, I, I, P, P,
                                                  P, P, P, P, P, P, Z, P]
        l.spec_verify_sample_filtered.restype = I
        l.spec_verify_typical.argtypes = [P, P, P, F, F, F, P, P, I, I, I, I, P, P, P, P, P, P, P,
                                          Z, P]
        l.spec_verify_typical.restype = I
        l.spec_verify_tree_workspace_size.argtypes = [I, I, I]
        l.spec_verify_tree_workspace_size.restype = Z
        l.spec_verify_tree_typical.argtypes = [P, P, I, P, P, F, F, F, P, P, I, I, I, I, I, P, P, P,
                                               Z, P]
        l.spec_verify_tree_sample.argtypes = [P, P, I, P, P, F, P, P, I, I, I, I, I, P, P, P, Z, P]
        l.spec_verify_tree_sample.restype = I
        l.spec_verify_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        l.spec_verify_set_wait_limit_ns.restype = I
        l.spec_verify_wait_limit_ns.argtypes = []
        l.spec_verify_wait_limit_ns.restype = ctypes.c_uint64
        l.spec_verify_tree_typical.restype = I
        l.spec_ngram_propose.argtypes = [P, P, I, I, I, I, I, P, P, P, P, P]
        l.spec_ngram_propose.restype = I
        l.spec_verify_tree.argtypes = [P, P, I, P, P, P, I, I, I, I, I, P, P, P]
        l.spec_verify_tree.restype = I
        l.spec_verify_status_string.argtypes = [I]
        l.spec_verify_status_string.restype = ctypes.c_char_p
        l.spec_verify_version.argtypes = []
        l.spec_verify_version.restype = I
        _lib = l
        return l
