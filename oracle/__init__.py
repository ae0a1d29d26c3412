"""DFlash2 draft-head oracle (fp64, CPU): TEST INFRASTRUCTURE ONLY.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  The product library never calls it, and the two share no
code: this module wraps ``dflash2_oracle.c`` (plain C loops in double
precision) through ctypes.

Every function follows ggml-org/llama.cpp pull request #27342, "spec : add
DFlash2 support (local convolution + candidate selector)", section "Overview"
(the convolution and edge formulas); the readings taken where that text is
silent are listed at the top of ``dflash2_oracle.c``.

Parity is pinned (not self-checked) by ``tests/test_oracle_pins.py``: library
routines (numpy convolve / matmul), closed forms, invariants, a second brute
force formulation, and hand-worked fixtures under ``tests/golden/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dflash2_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, extra_flags: tuple = ()) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math) into liboracle.so."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", "-Wall", "-Wextra", "-Werror", *extra_flags, _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            L = ctypes.c_long
            lib.oracle_dynconv.argtypes = [dp, dp, dp, dp, dp, L, L, L, L, L]
            lib.oracle_dynconv.restype = ctypes.c_int
            lib.oracle_project.argtypes = [dp, dp, dp, L, L, L]
            lib.oracle_project.restype = None
            lib.oracle_edges.argtypes = [ip, dp, dp, dp, dp, L, L, L, L, L, dp, ip, dp]
            lib.oracle_edges.restype = ctypes.c_int
            lib.oracle_select.argtypes = [dp, dp, ip, dp, dp, dp, L, L, L, L, L, L,
                                          dp, dp, ip, dp]
            lib.oracle_select.restype = ctypes.c_int
            lib.oracle_topk.argtypes = [dp, L, L, L, ip, dp]
            lib.oracle_topk.restype = ctypes.c_int
            lib.oracle_chain.argtypes = [ip, dp, dp, ip, ip, L, L, L, ctypes.c_double, ip, dp, ip]
            lib.oracle_chain.restype = ctypes.c_int
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _dp(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def max_threads() -> int:
    """OpenMP threads the oracle runs on."""
    return int(_load().oracle_max_threads())


def dynconv(x, hist, base, delta):
    """out[S,n,C] (float64) of the grouped dynamic depthwise causal conv.

    x [S,n,C]; hist [S,T-1,C] or None (zeros); base [T,C]; delta [S,n,T,G].
    """
    x = _f64(x)
    S, n, C = x.shape
    base = _f64(base)
    T = base.shape[0]
    delta = _f64(delta)
    G = delta.shape[-1]
    assert base.shape == (T, C) and delta.shape == (S, n, T, G)
    h = None
    if hist is not None:
        h = _f64(hist)
        assert h.shape == (S, T - 1, C)
        if T == 1:
            h = np.zeros((1,), np.float64)  # never read when T == 1
    out = np.empty((S, n, C), np.float64)
    rc = _load().oracle_dynconv(_dp(x), _dp(h), _dp(base), _dp(delta), _dp(out),
                                S, n, C, T, G)
    if rc != 0:
        raise ValueError("oracle_dynconv: C must be a multiple of G")
    return out


def project(h, W):
    """u[P,R] = h[P,d] W[R,d]^T in float64."""
    h = _f64(h)
    W = _f64(W)
    P, d = h.shape
    R = W.shape[0]
    assert W.shape == (R, d)
    u = np.empty((P, R), np.float64)
    _load().oracle_project(_dp(h), _dp(W), _dp(u), P, d, R)
    return u


def edges(cand_ids, u, A, B, unary, want_edges=True):
    """(edges [S,n-1,K,K] or None, best_slot [S,n-1,K], best_score [S,n-1,K]).

    cand_ids, unary [S,n,K]; u [S*n,R]; A, B [V,R].
    """
    cand_ids = _i32(cand_ids)
    S, n, K = cand_ids.shape
    A = _f64(A)
    B = _f64(B)
    V, R = A.shape
    u = _f64(u).reshape(S * n, R)
    unary = _f64(unary)
    assert B.shape == (V, R) and unary.shape == (S, n, K)
    E = max(n - 1, 0)
    e = np.empty((S, E, K, K), np.float64) if want_edges else None
    slot = np.empty((S, E, K), np.int32)
    score = np.empty((S, E, K), np.float64)
    rc = _load().oracle_edges(_ip(cand_ids), _dp(u), _dp(A), _dp(B), _dp(unary),
                              S, n, K, R, V, _dp(e), _ip(slot), _dp(score))
    if rc != 0:
        raise ValueError("oracle_edges: candidate id outside [0, V)")
    return e, slot, score


def select(h, W, cand_ids, A, B, unary, want_edges=True):
    """Composite selector: (u, edges, best_slot, best_score)."""
    cand_ids = _i32(cand_ids)
    S, n, K = cand_ids.shape
    h = _f64(h).reshape(S * n, -1)
    d = h.shape[1]
    W = _f64(W)
    R = W.shape[0]
    A = _f64(A)
    B = _f64(B)
    V = A.shape[0]
    unary = _f64(unary)
    u = np.empty((S * n, R), np.float64)
    E = max(n - 1, 0)
    e = np.empty((S, E, K, K), np.float64) if want_edges else None
    slot = np.empty((S, E, K), np.int32)
    score = np.empty((S, E, K), np.float64)
    rc = _load().oracle_select(_dp(h), _dp(W), _ip(cand_ids), _dp(A), _dp(B), _dp(unary),
                               S, n, d, K, R, V, _dp(u), _dp(e), _ip(slot), _dp(score))
    if rc != 0:
        raise ValueError("oracle_select: candidate id outside [0, V)")
    return u, e, slot, score


def topk(z, K):
    """(ids [rows,K] int32, vals [rows,K] float64): the K largest of each row of
    z [rows,V], descending, ties by ascending index."""
    z = _f64(z)
    rows, V = z.shape
    ids = np.empty((rows, K), np.int32)
    vals = np.empty((rows, K), np.float64)
    if _load().oracle_topk(_dp(z), rows, V, K, _ip(ids), _dp(vals)) != 0:
        raise ValueError("oracle_topk: need 1 <= K <= V")
    return ids, vals


def chain(cand_ids, unary, edges, best_slot, p_min, start_slot=None):
    """(tokens [S,n] int32, probs [S,n] float64, length [S] int32) of the greedy
    chain through each sequence's argmax table, cut at the first p < p_min.

    cand_ids, unary [S,n,K]; edges [S,n-1,K,K]; best_slot [S,n-1,K];
    start_slot [S] (a slot, or -1 for the unary argmax) or None.
    """
    cand_ids = _i32(cand_ids)
    S, n, K = cand_ids.shape
    unary = _f64(unary)
    E = max(n - 1, 0)
    edges = _f64(edges).reshape(S, E, K, K) if E else np.zeros((1,), np.float64)
    best_slot = _i32(best_slot).reshape(S, E, K) if E else np.zeros((1,), np.int32)
    st = None if start_slot is None else _i32(start_slot)
    tokens = np.empty((S, n), np.int32)
    probs = np.empty((S, n), np.float64)
    length = np.empty((S,), np.int32)
    rc = _load().oracle_chain(_ip(cand_ids), _dp(unary), _dp(edges), _ip(best_slot),
                              _ip(st) if st is not None else ctypes.POINTER(ctypes.c_int32)(),
                              S, n, K, float(p_min), _ip(tokens), _dp(probs), _ip(length))
    if rc != 0:
        raise ValueError("oracle_chain: slot outside [0, K)")
    return tokens, probs, length


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
