"""ctypes binding of libdflash2.so (the C ABI declared in include/dflash2.h).

Argument marshalling only: shapes and dtypes are read from torch tensors,
outputs are allocated with torch when the caller does not pass them, and the
call goes to the CUDA library on the tensors' current stream.  There is no
fallback: if the library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdflash2.so")

DF2_OK, DF2_ERR_INVALID_ARG, DF2_ERR_UNSUPPORTED, DF2_ERR_CUDA = 0, 1, 2, 3
DF2_F32, DF2_BF16 = 0, 1
FLAG_BAD_ID, FLAG_TIMEOUT, FLAG_OVERFLOW = 1, 2, 4

_lock = threading.Lock()
_lib = None


class Dflash2Error(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it first "
                    "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            vp, i = ctypes.c_void_p, ctypes.c_int
            L.dflash2_version.argtypes = []
            L.dflash2_version.restype = i
            L.dflash2_status_string.argtypes = [i]
            L.dflash2_status_string.restype = ctypes.c_char_p
            L.dflash2_last_error.argtypes = []
            L.dflash2_last_error.restype = ctypes.c_char_p
            L.dflash2_dynconv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp]
            L.dflash2_dynconv.restype = i
            L.dflash2_project.argtypes = [vp, vp, vp, i, i, i, i, vp]
            L.dflash2_project.restype = i
            L.dflash2_project_workspace_bytes.argtypes = [i, i, i]
            L.dflash2_project_workspace_bytes.restype = ctypes.c_size_t
            L.dflash2_project_ws.argtypes = [vp, vp, vp, i, i, i, i, vp, ctypes.c_size_t, vp]
            L.dflash2_project_ws.restype = i
            L.dflash2_project_noalloc.argtypes = [vp, vp, vp, i, i, i, i, vp]
            L.dflash2_project_noalloc.restype = i
            L.dflash2_edges.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, vp, vp, vp, vp, vp]
            L.dflash2_edges.restype = i
            L.dflash2_select.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp, vp, vp,
                                         vp, vp, vp]
            L.dflash2_select.restype = i
            L.dflash2_predict_delta.argtypes = [vp, vp, vp, i, i, i, i, vp]
            L.dflash2_predict_delta.restype = i
            L.dflash2_dynconv_predicted.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp]
            L.dflash2_dynconv_predicted.restype = i
            L.dflash2_chain.argtypes = [vp, vp, vp, vp, vp, i, i, i, ctypes.c_float, vp, vp, vp,
                                        vp, vp]
            L.dflash2_chain.restype = i
            L.dflash2_topk.argtypes = [vp, i, i, i, i, vp, vp, vp]
            L.dflash2_topk.restype = i
            L.dflash2_select_plan.argtypes = [i, i, i, i, i, i, ctypes.POINTER(ctypes.c_int)]
            L.dflash2_select_plan.restype = i
            L.dflash2_probe_gather.argtypes = [vp, ctypes.c_longlong, i, vp, i, vp, vp]
            L.dflash2_probe_gather.restype = i
            L.dflash2_take_device_faults.argtypes = [ctypes.POINTER(ctypes.c_int32)]
            L.dflash2_take_device_faults.restype = i
            _lib = L
    return _lib


def _check(status: int):
    if status != DF2_OK:
        L = lib()
        raise Dflash2Error(status, f"{L.dflash2_status_string(status).decode()}: "
                                   f"{L.dflash2_last_error().decode()}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(dev) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)


def _code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return DF2_BF16
    if dt == torch.float32:
        return DF2_F32
    raise TypeError(f"unsupported dtype {dt}")


def _need(t, name, dtype=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def version() -> int:
    return lib().dflash2_version()


def dynconv(x, hist, base, delta, out=None, out_dtype=None):
    """Grouped dynamic depthwise causal conv: x [S,n,C], hist [S,T-1,C] or None,
    base [T,C], delta [S,n,T,G] -> out [S,n,C]."""
    S, n, C = x.shape
    T = base.shape[0]
    G = delta.shape[-1]
    for t, nm in ((x, "x"), (hist, "hist"), (base, "base"), (delta, "delta")):
        _need(t, nm, x.dtype)
    if out is None:
        out = torch.empty((S, n, C), dtype=out_dtype or x.dtype, device=x.device)
    _need(out, "out")
    _check(lib().dflash2_dynconv(_ptr(x), _ptr(hist), _ptr(base), _ptr(delta), _ptr(out),
                                 S, n, C, T, G, _code(x.dtype), _code(out.dtype),
                                 _stream(x.device)))
    return out


def project_workspace_bytes(P: int, d: int, R: int) -> int:
    """Bytes of split-K workspace project(..., workspace=...) needs on this device."""
    return int(lib().dflash2_project_workspace_bytes(P, d, R))


def project(h, W, u=None, workspace=None):
    """u [P,R] fp32 = h [P,d] @ W[R,d]^T.  With `workspace` (a CUDA tensor of at
    least project_workspace_bytes(P, d, R) bytes) the split-K partial tiles are
    exchanged through it instead of through distributed shared memory."""
    P, d = h.shape
    R = W.shape[0]
    _need(h, "h")
    _need(W, "W", h.dtype)
    if u is None:
        u = torch.empty((P, R), dtype=torch.float32, device=h.device)
    _need(u, "u", torch.float32)
    if workspace is None:
        _check(lib().dflash2_project(_ptr(h), _ptr(W), _ptr(u), P, d, R, _code(h.dtype),
                                     _stream(h.device)))
    else:
        _need(workspace, "workspace")
        _check(lib().dflash2_project_ws(_ptr(h), _ptr(W), _ptr(u), P, d, R, _code(h.dtype),
                                        _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        _stream(h.device)))
    return u


def project_noalloc(h, W, u=None):
    """project() through the library's fixed workspace (no device allocation by
    the library; u must be passed to avoid torch allocating it)."""
    P, d = h.shape
    R = W.shape[0]
    _need(h, "h")
    _need(W, "W", h.dtype)
    if u is None:
        u = torch.empty((P, R), dtype=torch.float32, device=h.device)
    _need(u, "u", torch.float32)
    _check(lib().dflash2_project_noalloc(_ptr(h), _ptr(W), _ptr(u), P, d, R, _code(h.dtype),
                                         _stream(h.device)))
    return u


def _edge_outputs(S, n, K, dev, edges_out, best_slot, best_score):
    E = max(n - 1, 0)
    if edges_out is True:
        edges_out = torch.empty((S, E, K, K), dtype=torch.float32, device=dev)
    elif edges_out is False:
        edges_out = None
    if best_slot is None:
        best_slot = torch.empty((S, E, K), dtype=torch.int32, device=dev)
    if best_score is None:
        best_score = torch.empty((S, E, K), dtype=torch.float32, device=dev)
    return edges_out, best_slot, best_score


def edges(cand_ids, u, A, B, unary, edges_out=None, best_slot=None, best_score=None,
          err_flag=None):
    """Edge scores + per-predecessor argmax.  cand_ids [S,n,K] int32, u [S*n,R] fp32,
    A, B [V,R], unary [S,n,K] fp32.  edges_out=True allocates the [S,n-1,K,K] matrix.
    Returns (edges_out or None, best_slot [S,n-1,K] int32, best_score [S,n-1,K] fp32)."""
    S, n, K = cand_ids.shape
    V, R = A.shape
    _need(cand_ids, "cand_ids", torch.int32)
    _need(u, "u", torch.float32)
    _need(A, "A")
    _need(B, "B", A.dtype)
    _need(unary, "unary", torch.float32)
    edges_out, best_slot, best_score = _edge_outputs(S, n, K, u.device, edges_out, best_slot,
                                                     best_score)
    _need(err_flag, "err_flag", torch.int32)
    _check(lib().dflash2_edges(_ptr(cand_ids), _ptr(u), _ptr(A), _ptr(B), _ptr(unary), S, n, K,
                               R, V, _code(A.dtype), _ptr(edges_out), _ptr(best_slot),
                               _ptr(best_score), _ptr(err_flag), _stream(u.device)))
    return edges_out, best_slot, best_score


def select(h, W, cand_ids, A, B, unary, u_out=None, edges_out=None, best_slot=None,
           best_score=None, err_flag=None):
    """Composite selector: project then edges.  h [S*n,d].
    Returns (u [S*n,R], edges_out or None, best_slot, best_score)."""
    S, n, K = cand_ids.shape
    d = h.shape[-1]
    V, R = A.shape
    _need(h, "h")
    _need(W, "W", h.dtype)
    _need(cand_ids, "cand_ids", torch.int32)
    _need(A, "A", h.dtype)
    _need(B, "B", h.dtype)
    _need(unary, "unary", torch.float32)
    if u_out is None:
        u_out = torch.empty((S * n, R), dtype=torch.float32, device=h.device)
    _need(u_out, "u_out", torch.float32)
    edges_out, best_slot, best_score = _edge_outputs(S, n, K, h.device, edges_out, best_slot,
                                                     best_score)
    _need(err_flag, "err_flag", torch.int32)
    _check(lib().dflash2_select(_ptr(h), _ptr(W), _ptr(cand_ids), _ptr(A), _ptr(B), _ptr(unary),
                                S, n, d, K, R, V, _code(h.dtype), _ptr(u_out), _ptr(edges_out),
                                _ptr(best_slot), _ptr(best_score), _ptr(err_flag),
                                _stream(h.device)))
    return u_out, edges_out, best_slot, best_score


def topk(logits, K, cand_ids=None, values=None):
    """Top-K candidates of every row: logits [..., V] (fp32 or bf16) ->
    (cand_ids [..., K] int32, values [..., K] fp32), descending, ties by index."""
    V = logits.shape[-1]
    lead = tuple(logits.shape[:-1])
    rows = 1
    for s in lead:
        rows *= s
    _need(logits, "logits")
    if cand_ids is None:
        cand_ids = torch.empty(lead + (K,), dtype=torch.int32, device=logits.device)
    if values is None:
        values = torch.empty(lead + (K,), dtype=torch.float32, device=logits.device)
    _need(cand_ids, "cand_ids", torch.int32)
    _need(values, "values", torch.float32)
    _check(lib().dflash2_topk(_ptr(logits), rows, V, K, _code(logits.dtype), _ptr(cand_ids),
                              _ptr(values), _stream(logits.device)))
    return cand_ids, values


def predict_delta(x, Wc, T, G, delta=None):
    """delta [S,n,T,G] = x [S,n,C] . Wc[T*G, C]^T in x's dtype (the conv's
    dynamic taps predicted from its input)."""
    S, n, C = x.shape
    _need(x, "x")
    _need(Wc, "Wc", x.dtype)
    if delta is None:
        delta = torch.empty((S, n, T, G), dtype=x.dtype, device=x.device)
    _need(delta, "delta", x.dtype)
    _check(lib().dflash2_predict_delta(_ptr(x), _ptr(Wc), _ptr(delta), S * n, C, T * G,
                                       _code(x.dtype), _stream(x.device)))
    return delta


def dynconv_predicted(x, hist, base, Wc, G, out=None, out_dtype=None):
    """The conv with its taps predicted from its input, fused: x [S,n,C], hist
    [S,T-1,C] or None, base [T,C], Wc [T*G,C] (bf16) -> out [S,n,C]; the same as
    dynconv(x, hist, base, predict_delta(x, Wc, T, G)) without delta in HBM."""
    S, n, C = x.shape
    T = base.shape[0]
    for t, nm in ((x, "x"), (hist, "hist"), (base, "base"), (Wc, "Wc")):
        _need(t, nm, x.dtype)
    if out is None:
        out = torch.empty((S, n, C), dtype=out_dtype or x.dtype, device=x.device)
    _need(out, "out")
    _check(lib().dflash2_dynconv_predicted(_ptr(x), _ptr(hist), _ptr(base), _ptr(Wc), _ptr(out),
                                           S, n, C, T, G, _code(x.dtype), _code(out.dtype),
                                           _stream(x.device)))
    return out


def chain(cand_ids, unary, edges, best_slot, p_min, start_slot=None, err_flag=None):
    """Greedy chain readout: (tokens [S,n] int32, probs [S,n] fp32, length [S] int32).
    cand_ids, unary [S,n,K]; edges [S,n-1,K,K] and best_slot [S,n-1,K] from
    select(..., edges_out=True) (None when n == 1); start_slot [S] int32 or None."""
    S, n, K = cand_ids.shape
    _need(cand_ids, "cand_ids", torch.int32)
    _need(unary, "unary", torch.float32)
    _need(edges, "edges", torch.float32)
    _need(best_slot, "best_slot", torch.int32)
    _need(start_slot, "start_slot", torch.int32)
    _need(err_flag, "err_flag", torch.int32)
    dev = cand_ids.device
    tokens = torch.empty((S, n), dtype=torch.int32, device=dev)
    probs = torch.empty((S, n), dtype=torch.float32, device=dev)
    length = torch.empty((S,), dtype=torch.int32, device=dev)
    _check(lib().dflash2_chain(_ptr(cand_ids), _ptr(unary), _ptr(edges), _ptr(best_slot),
                               _ptr(start_slot), S, n, K, float(p_min), _ptr(tokens), _ptr(probs),
                               _ptr(length), _ptr(err_flag), _stream(dev)))
    return tokens, probs, length


def take_device_faults() -> int:
    """Read and clear the library's device fault word (synchronises the device)."""
    v = ctypes.c_int32(0)
    _check(lib().dflash2_take_device_faults(ctypes.byref(v)))
    return int(v.value)


def probe_gather(table, row_bytes: int, ids, out=None):
    """Measurement aid: out[i] (int32 view of a uint32) = XOR of the 32-bit words of
    row ids[i] of `table` viewed as [rows, row_bytes] bytes."""
    _need(table, "table")
    _need(ids, "ids", torch.int32)
    nbytes = table.numel() * table.element_size()
    rows = nbytes // int(row_bytes)
    n_ids = ids.numel()
    if out is None:
        out = torch.empty((n_ids,), dtype=torch.int32, device=ids.device)
    _need(out, "out", torch.int32)
    _check(lib().dflash2_probe_gather(_ptr(table), rows, int(row_bytes), _ptr(ids), n_ids,
                                      _ptr(out), _stream(ids.device)))
    return out


def select_plan(S: int, n: int, d: int, K: int, R: int, dtype=torch.bfloat16) -> dict:
    """How select() runs these shapes on the current device: {"fused": bool,
    "cluster_size", "clusters", "rows_per_block"}."""
    out = (ctypes.c_int * 4)()
    _check(lib().dflash2_select_plan(S, n, d, K, R, _code(dtype), out))
    return {"fused": bool(out[0]), "cluster_size": out[1], "clusters": out[2],
            "rows_per_block": out[3]}
