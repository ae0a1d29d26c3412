"""The C ABI library builds, loads and exports every declared entry point; host-side
argument validation rejects bad calls before anything is launched (CPU only:
every call here fails validation, so no CUDA work is issued)."""
import ctypes
import os
import re

import pytest

from dflash2_draft_head_gb300 import binding, build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash2.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash2_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def L():
    build_library()
    return binding.lib()


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 8
    for n in names:
        assert hasattr(L, n), n
        assert ctypes.cast(getattr(L, n), ctypes.c_void_p).value


def test_version_and_status_strings(L):
    assert L.dflash2_version() >= 100
    for code, name in [(0, b"DF2_OK"), (1, b"DF2_ERR_INVALID_ARG"), (2, b"DF2_ERR_UNSUPPORTED"),
                       (3, b"DF2_ERR_CUDA")]:
        assert L.dflash2_status_string(code) == name
    assert L.dflash2_status_string(99) == b"DF2_UNKNOWN_STATUS"


# fake, 16-byte aligned, non-overlapping addresses: only ever passed to calls
# that must fail validation before any launch
P = [ctypes.c_void_p(0x10000000 * (k + 1)) for k in range(12)]
NULL = None


def _dyn(L, x=P[0], hist=P[1], base=P[2], delta=P[3], out=P[4], S=2, n=8, C=64, T=4, G=4,
         di=1, do=1):
    return L.dflash2_dynconv(x, hist, base, delta, out, S, n, C, T, G, di, do, None)


@pytest.mark.parametrize("kw,code", [
    (dict(x=NULL), 1), (dict(out=NULL), 1), (dict(base=NULL), 1), (dict(delta=NULL), 1),
    (dict(S=0), 1), (dict(n=-1), 1), (dict(C=0), 1), (dict(T=0), 1), (dict(G=0), 1),
    (dict(C=64, G=5), 1), (dict(di=7), 1), (dict(x=ctypes.c_void_p(0x10000008)), 1),
    (dict(out=P[0]), 1),                       # out aliases x
    (dict(C=60, G=4), 2),                      # C % 8
    (dict(C=64, G=16), 2),                     # C/G = 4
    (dict(T=17), 2), (dict(di=0, do=1), 2),
])
def test_dynconv_validation(L, kw, code):
    assert _dyn(L, **kw) == code
    assert L.dflash2_last_error()


def test_dynconv_hist_overlapping_out_is_rejected(L):
    # hist [2,3,64] bf16 = 768 B placed 256 B before out: overlaps
    out = ctypes.c_void_p(0x50000000)
    hist = ctypes.c_void_p(0x50000000 - 256)
    assert _dyn(L, hist=hist, out=out) == 1


def _proj(L, h=P[0], W=P[1], u=P[2], Pn=16, d=64, R=16, dt=1):
    return L.dflash2_project(h, W, u, Pn, d, R, dt, None)


@pytest.mark.parametrize("kw,code", [
    (dict(h=NULL), 1), (dict(u=NULL), 1), (dict(Pn=0), 1), (dict(d=0), 1), (dict(R=0), 1),
    (dict(dt=3), 1), (dict(u=P[0]), 1), (dict(W=ctypes.c_void_p(0x20000004)), 1),
    (dict(R=12), 2), (dict(R=520), 2), (dict(d=36), 2),
])
def test_project_validation(L, kw, code):
    assert _proj(L, **kw) == code


def _edges(L, ids=P[0], u=P[1], A=P[2], B=P[3], un=P[4], S=2, n=4, K=4, R=16, V=100, dt=1,
           eo=P[5], bs=P[6], bsc=P[7], flag=P[8]):
    return L.dflash2_edges(ids, u, A, B, un, S, n, K, R, V, dt, eo, bs, bsc, flag, None)


@pytest.mark.parametrize("kw,code", [
    (dict(ids=NULL), 1), (dict(A=NULL), 1), (dict(bs=NULL), 1), (dict(bsc=NULL), 1),
    (dict(S=0), 1), (dict(K=0), 1), (dict(V=0), 1), (dict(R=-8), 1), (dict(dt=2), 1),
    (dict(bs=P[0]), 1), (dict(eo=P[2]), 1), (dict(bsc=P[6]), 1),
    (dict(flag=ctypes.c_void_p(0x90000002)), 1),
    (dict(K=257), 2), (dict(R=20), 2), (dict(R=528), 2),
])
def test_edges_validation(L, kw, code):
    assert _edges(L, **kw) == code


def test_select_validation(L):
    args = [P[0], P[1], P[2], P[3], P[4], P[5], 2, 4, 64, 4, 16, 100, 1, P[6], P[7], P[8], P[9],
            P[10], None]
    a = list(args)
    a[13] = P[0]  # u_out aliases h
    assert L.dflash2_select(*a) == 1
    a = list(args)
    a[13] = P[3]  # u_out aliases A
    assert L.dflash2_select(*a) == 1
    a = list(args)
    a[6] = 0
    assert L.dflash2_select(*a) == 1
    a = list(args)
    a[10] = 12
    assert L.dflash2_select(*a) == 2


def test_take_device_faults_rejects_null(L):
    assert L.dflash2_take_device_faults(None) == 1


def test_project_ws_validation(L):
    L.dflash2_project_workspace_bytes.restype = ctypes.c_size_t
    L.dflash2_project_workspace_bytes.argtypes = [ctypes.c_int] * 3
    need = L.dflash2_project_workspace_bytes(4096, 5120, 128)
    assert need > 0 and need % 16 == 0
    assert L.dflash2_project_workspace_bytes(0, 5120, 128) == 0
    f = L.dflash2_project_ws
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_void_p, ctypes.c_size_t,
                                                               ctypes.c_void_p]
    args = [P[0], P[1], P[2], 4096, 5120, 128, 1]
    assert f(*args, None, 0, None) == 1                       # workspace missing
    assert f(*args, P[3], need - 16, None) == 1               # workspace too small
    assert f(*args, ctypes.c_void_p(0x40000008), need, None) == 1  # misaligned
    assert f(*args, P[0], need, None) == 1                    # overlaps h
    assert b"workspace" in L.dflash2_last_error()
    assert f(P[0], P[1], P[2], 4096, 5120, 12, 1, P[3], need, None) == 2  # R % 8


def _topk(L, lg=P[0], rows=4, V=100, K=8, dt=0, ids=P[1], vals=P[2]):
    return L.dflash2_topk(lg, rows, V, K, dt, ids, vals, None)


@pytest.mark.parametrize("kw,code", [
    (dict(lg=NULL), 1), (dict(ids=NULL), 1), (dict(vals=NULL), 1),
    (dict(rows=0), 1), (dict(V=0), 1), (dict(K=0), 1), (dict(K=101), 1), (dict(dt=2), 1),
    (dict(lg=ctypes.c_void_p(0x10000004)), 1), (dict(vals=ctypes.c_void_p(0x30000008)), 1),
    (dict(ids=P[0]), 1),                        # cand_ids aliases the logits
    (dict(vals=P[1]), 1),                       # the two outputs alias
    (dict(V=5000, K=1025), 2),
])
def test_topk_validation(L, kw, code):
    assert _topk(L, **kw) == code
    assert b"topk" in L.dflash2_last_error() or b"aligned" in L.dflash2_last_error() or \
        b"overlaps" in L.dflash2_last_error()


def _chain(L, ci=P[0], un=P[1], ed=P[2], bs=P[3], st=None, S=2, n=4, K=8, pm=0.5, tk=P[4],
           pr=P[5], ln=P[6], fl=None):
    f = L.dflash2_chain
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 3 + [ctypes.c_float] + \
        [ctypes.c_void_p] * 5
    return f(ci, un, ed, bs, st, S, n, K, pm, tk, pr, ln, fl, None)


@pytest.mark.parametrize("kw,code", [
    (dict(ci=NULL), 1), (dict(tk=NULL), 1), (dict(ln=NULL), 1), (dict(ed=NULL), 1),
    (dict(bs=NULL), 1), (dict(S=0), 1), (dict(n=0), 1), (dict(K=-1), 1),
    (dict(tk=P[0]), 1),                              # tokens alias cand_ids
    (dict(pr=ctypes.c_void_p(0x60000004)), 1),       # misaligned
    (dict(fl=ctypes.c_void_p(0x70000002)), 1),       # err_flag not 4-byte aligned
    (dict(n=7000, K=8), 2),                          # argmax table above 200 KB
])
def test_chain_validation(L, kw, code):
    assert _chain(L, **kw) == code
    assert L.dflash2_last_error()


def test_chain_single_position_needs_no_table(L):
    # n == 1: edges and best_slot may be NULL; the call then fails only on a bad size
    assert _chain(L, ed=NULL, bs=NULL, n=1, S=0) == 1


def _pdelta(L, x=P[0], wc=P[1], de=P[2], Pn=64, C=128, TG=16, dt=1):
    return L.dflash2_predict_delta(x, wc, de, Pn, C, TG, dt, None)


@pytest.mark.parametrize("kw,code", [
    (dict(x=NULL), 1), (dict(de=NULL), 1), (dict(Pn=0), 1), (dict(C=-1), 1), (dict(TG=0), 1),
    (dict(dt=5), 1), (dict(de=P[0]), 1), (dict(wc=ctypes.c_void_p(0x20000002)), 1),
    (dict(TG=12), 2), (dict(TG=520), 2), (dict(C=100), 2),
])
def test_predict_delta_validation(L, kw, code):
    assert _pdelta(L, **kw) == code


def _dpred(L, x=P[0], hist=P[1], base=P[2], wc=P[3], out=P[4], S=2, n=8, C=64, T=4, G=4,
           di=1, do=1):
    return L.dflash2_dynconv_predicted(x, hist, base, wc, out, S, n, C, T, G, di, do, None)


@pytest.mark.parametrize("kw,code", [
    (dict(x=NULL), 1), (dict(wc=NULL), 1), (dict(base=NULL), 1), (dict(out=NULL), 1),
    (dict(S=0), 1), (dict(n=-1), 1), (dict(C=0), 1), (dict(T=0), 1), (dict(G=0), 1),
    (dict(C=64, G=5), 1), (dict(di=7), 1), (dict(do=3), 1),
    (dict(x=ctypes.c_void_p(0x10000008)), 1),
    (dict(out=P[0]), 1),                       # out aliases x
    (dict(out=P[3]), 1),                       # out aliases Wc
    (dict(di=0, do=1), 2),                     # fp32 input with bf16 output
    (dict(T=9, G=8), 2),                       # T > 8
    (dict(C=60, G=4), 2),                      # C % 8
    (dict(C=64, G=16), 2),                     # C/G = 4
    (dict(T=3, G=4), 2),                       # T*G = 12
    (dict(C=2048, T=8, G=64), 2),              # T*G = 512
])
def test_dynconv_predicted_validation(L, kw, code):
    assert _dpred(L, **kw) == code
    assert L.dflash2_last_error()


def _probe(L, tb=P[0], rows=1000, rb=256, ids=P[1], n=64, out=P[2]):
    return L.dflash2_probe_gather(tb, rows, rb, ids, n, out, None)


@pytest.mark.parametrize("kw,code", [
    (dict(tb=NULL), 1), (dict(ids=NULL), 1), (dict(out=NULL), 1), (dict(rows=0), 1),
    (dict(n=-1), 1), (dict(rb=8), 1), (dict(rb=96), 1), (dict(rb=1024), 1),
    (dict(tb=ctypes.c_void_p(0x10000004)), 1),
    (dict(out=P[0]), 1),                       # out inside the table
])
def test_probe_gather_validation(L, kw, code):
    assert _probe(L, **kw) == code
    assert L.dflash2_last_error()


def test_trace_read_is_unsupported_without_tracing(L):
    """The normal library has no trace table: the call reports it and touches no device."""
    buf = (ctypes.c_uint64 * 4)()
    L.dflash2_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
    assert L.dflash2_trace_read(ctypes.addressof(buf), 32, 0) == 2


def test_topk_trace_read_is_unsupported_without_tracing(L):
    buf = (ctypes.c_uint64 * 4)()
    L.dflash2_trace_read_topk.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
    assert L.dflash2_trace_read_topk(ctypes.addressof(buf), 32, 0) == 2
