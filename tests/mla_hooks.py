"""ctypes binding of the test-only hooks library tests/hooks/libmla_debug.so
(declared in tests/hooks/mla_debug.h): single kernels of the MLA library
exposed for the tests.  libmla.so itself carries no test entry points."""
from __future__ import annotations

import ctypes
import os

HOOKS_LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "hooks", "libmla_debug.so")

_VP, _I = ctypes.c_void_p, ctypes.c_int
_SIGS = {
    "mla_debug_gemm": (_I, [_VP, _I, _VP, _I, _I, _VP, _I, _I, _I, _I, _VP]),
    "mla_debug_wait_timeout": (_I, [_VP, ctypes.c_uint64, _VP]),
    "mla_debug_umma_probe": (_I, [_VP, _I, _VP]),
}
_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(HOOKS_LIB):
            raise RuntimeError(f"{HOOKS_LIB} not found: build with __graft_entry__.build()")
        L = ctypes.CDLL(HOOKS_LIB)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(rc, where):
    if rc != 0:
        raise RuntimeError(f"{where}: status {rc}")


def mla_debug_gemm(A, B, C, b_mn_major=False):
    """C = A @ B^T (B [N, K]) or A @ B (B [K, N] when b_mn_major)."""
    M, K = A.shape
    N = B.shape[0] if not b_mn_major else B.shape[1]
    _check(lib().mla_debug_gemm(_ptr(A), A.stride(0), _ptr(B), B.stride(0), int(b_mn_major), _ptr(C), C.stride(0),
                                M, N, K, _stream()), "mla_debug_gemm")


def mla_debug_wait_timeout(status_word, limit_ns: int):
    _check(lib().mla_debug_wait_timeout(_ptr(status_word), limit_ns, _stream()), "mla_debug_wait_timeout")


def mla_debug_umma_probe(out, m: int):
    _check(lib().mla_debug_umma_probe(_ptr(out), m, _stream()), "mla_debug_umma_probe")
