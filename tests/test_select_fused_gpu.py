"""The one-kernel selector (dflash2_select on bf16 shapes it takes) against the
fp64 oracle: u, the full edge matrix, best score and the argmax rule, on shapes
chosen to cross every boundary of its decomposition: cluster sizes from the
planner, row blocks that cut sequences, several waves of row blocks per
cluster, ragged last tiles, d not a multiple of 64, every supported K and R,
sequences of two positions, and out-of-range ids (clamped and flagged).
Each case first asserts that the fused kernel is the path that runs.
"""
import numpy as np
import pytest
import torch

import dflash2_draft_head_gb300 as df2
import oracle
from dflash2_draft_head_gb300 import synth
from dflash2_draft_head_gb300.workloads import Workload
from helpers import assert_argmax, assert_close, dev, host

pytestmark = pytest.mark.gpu


def W_(S, n, d, K, R, V, seed=11):
    return Workload(name="fused_case", S=S, n=n, C=64, T=4, G=4, d=d, R=R, V=V, K=K,
                    dtype="bf16", S_sel=S, n_sel=n, seed=seed)


def run(w, ids=None, with_edges=True, flag=None):
    cb = synth.codebooks(w)
    sel = synth.selector_inputs(w)
    cand = sel["cand_ids"] if ids is None else ids
    u, e, slot, score = df2.select(dev(sel["h"], "bf16"), dev(cb["W"], "bf16"), dev(cand),
                                   dev(cb["A"], "bf16"), dev(cb["B"], "bf16"),
                                   dev(sel["unary"]), edges_out=with_edges, err_flag=flag)
    torch.cuda.synchronize()
    return cb, sel, u, e, slot, score


def check(w, with_edges=True):
    plan = df2.select_plan(w.S_sel, w.n_sel, w.d, w.K, w.R)
    assert plan["fused"], plan
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    cb, sel, u, e, slot, score = run(w, with_edges=with_edges, flag=flag)
    assert int(flag.item()) == 0
    assert df2.take_device_faults() == 0
    u_o, e_o, slot_o, score_o = oracle.select(sel["h"].numpy(), cb["W"].numpy(),
                                              sel["cand_ids"].numpy(), cb["A"].numpy(),
                                              cb["B"].numpy(), sel["unary"].numpy())
    assert_close(host(u), u_o, "bf16", "fused u")
    if with_edges:
        assert_close(host(e), e_o, "bf16", "fused edges")
    assert_close(host(score), score_o, "bf16", "fused best_score")
    assert_argmax(host(slot), e_o, slot_o, "bf16", "fused argmax")
    return plan


@pytest.mark.parametrize("S,n,d,K,R,V", [
    (3, 7, 256, 16, 128, 2000),       # small: up to 4 CTAs split d
    (2, 9, 5120, 16, 128, 151936),    # two draft blocks at Qwen-27B width
    (5, 5, 200, 8, 64, 1000),         # d % 64 != 0 (last k-block zero-filled), R = 64
    (4, 3, 384, 4, 64, 100),          # K = 4: 32 transitions per tile
    (3, 4, 512, 32, 128, 4000),       # K = 32
    (2, 5, 512, 64, 256, 5000),       # K = 64, R = 256: two edge stages per tile
    (2, 3, 640, 128, 256, 5000),      # K = 128: one transition per tile
    (37, 2, 256, 16, 128, 3000),      # n = 2: one transition per sequence
    (1, 300, 512, 8, 128, 1000),      # one long sequence: row blocks cut it
    (1024, 16, 128, 16, 64, 5000),    # 16384 rows: several row blocks per cluster
    (130, 3, 5376, 64, 256, 262144),  # Gemma width, ragged tiles
])
def test_fused_select_shapes(S, n, d, K, R, V):
    check(W_(S, n, d, K, R, V))


def test_fused_select_without_edge_matrix():
    check(W_(64, 16, 1024, 16, 128, 151936), with_edges=False)


def test_fused_select_bad_ids_are_clamped_and_flagged():
    w = W_(4, 6, 256, 16, 128, 640)
    sel = synth.selector_inputs(w)
    ids = sel["cand_ids"].clone()
    ids[0, 1, 2] = 640    # past the end -> row 639
    ids[3, 4, 9] = -3     # negative -> row 0
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    cb, sel, u, e, slot, score = run(w, ids=ids, flag=flag)
    assert int(flag.item()) & df2.binding.FLAG_BAD_ID
    u_o, e_o, _, _ = oracle.select(sel["h"].numpy(), cb["W"].numpy(), ids.clamp(0, 639).numpy(),
                                   cb["A"].numpy(), cb["B"].numpy(), sel["unary"].numpy())
    assert_close(host(e), e_o, "bf16", "fused edges with clamped ids")


def test_fused_matches_two_kernel_path():
    """The same shapes through dflash2_project + dflash2_edges (the path other
    shapes take) agree with the fused kernel within the bf16 tolerance."""
    w = W_(16, 16, 2048, 16, 128, 20000)
    cb, sel, u, e, slot, score = run(w)
    u2 = df2.project(dev(sel["h"], "bf16"), dev(cb["W"], "bf16"))
    e2, slot2, score2 = df2.edges(dev(sel["cand_ids"]), u2, dev(cb["A"], "bf16"),
                                  dev(cb["B"], "bf16"), dev(sel["unary"]), edges_out=True)
    torch.cuda.synchronize()
    assert_close(host(u), host(u2).astype(np.float64), "bf16", "fused vs two-kernel u")
    assert_close(host(e), host(e2).astype(np.float64), "bf16", "fused vs two-kernel edges")


def test_plan_reports_the_two_kernel_path_for_other_shapes():
    assert not df2.select_plan(4, 8, 256, 16, 96, torch.bfloat16)["fused"]   # R = 96
    assert not df2.select_plan(4, 8, 256, 3, 128, torch.bfloat16)["fused"]   # K = 3
    assert not df2.select_plan(4, 1, 256, 16, 128, torch.bfloat16)["fused"]  # n = 1
    assert not df2.select_plan(4, 8, 256, 16, 128, torch.float32)["fused"]   # fp32


def test_fused_select_repeated_calls_are_identical():
    """Deterministic: the split-d sums are reduced in a fixed order."""
    w = W_(32, 16, 5120, 16, 128, 151936)
    _, _, u1, e1, s1, _ = run(w)
    _, _, u2, e2, s2, _ = run(w)
    assert torch.equal(u1, u2) and torch.equal(e1, e2) and torch.equal(s1, s2)


@pytest.mark.parametrize("S,n,d,K,R,V", [
    (256, 16, 512, 16, 128, 151936),  # the batched shape's edge work (d shortened)
    (16, 8, 256, 64, 256, 4096),      # two units per tile (R = 256), K = 64
    (7, 5, 256, 4, 64, 500),          # K = 4, R = 64, ragged tiles
])
def test_edges_call_matches_the_selectors_edge_phase(S, n, d, K, R, V):
    """dflash2_edges on bf16 codebooks runs the selector's edge phase on the given u,
    with its own row decomposition (one CTA per cluster): given the selector's u it
    must reproduce the selector's edge scores, argmax and best scores exactly."""
    w = W_(S, n, d, K, R, V)
    cb, sel, u, e, slot, score = run(w)
    e2, slot2, score2 = df2.edges(dev(sel["cand_ids"]), u, dev(cb["A"], "bf16"),
                                  dev(cb["B"], "bf16"), dev(sel["unary"]), edges_out=True)
    torch.cuda.synchronize()
    assert torch.equal(e, e2) and torch.equal(slot, slot2) and torch.equal(score, score2)


@pytest.mark.gpu
def test_traced_build_matches_and_records_phases():
    """The selector built with its trace points gives the same outputs as the
    normal library, and each CTA's stamps are ordered along the kernel."""
    import ctypes
    from dflash2_draft_head_gb300 import build as B
    from dflash2_draft_head_gb300.workloads import BY_NAME
    w = BY_NAME["qwen27b_single_block16"]
    cb = synth.codebooks(w)
    si = synth.selector_inputs(w)
    bt = torch.bfloat16
    h, W, A, Bm = (t.to(bt).cuda() for t in (si["h"], cb["W"], cb["A"], cb["B"]))
    ids, un = si["cand_ids"].cuda(), si["unary"].cuda()
    u0, e0, s0, c0 = df2.select(h, W, ids, A, Bm, un)
    T = ctypes.CDLL(B.build_traced())
    vp = ctypes.c_void_p
    T.dflash2_trace_read.argtypes = [vp, ctypes.c_int, ctypes.c_int]
    P, E = w.S_sel * w.n_sel, w.S_sel * (w.n_sel - 1)
    u = torch.empty((P, w.R), dtype=torch.float32, device="cuda")
    slot = torch.empty((E, w.K), dtype=torch.int32, device="cuda")
    score = torch.empty((E, w.K), dtype=torch.float32, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    buf = torch.zeros(512 * 64, dtype=torch.int64)
    torch.cuda.synchronize()
    assert T.dflash2_trace_read(vp(buf.data_ptr()), buf.numel() * 8, 1) == 0
    rc = T.dflash2_select(vp(h.data_ptr()), vp(W.data_ptr()), vp(ids.data_ptr()), vp(A.data_ptr()),
                          vp(Bm.data_ptr()), vp(un.data_ptr()), w.S_sel, w.n_sel, w.d, w.K, w.R,
                          w.V, 1, vp(u.data_ptr()), None, vp(slot.data_ptr()), vp(score.data_ptr()),
                          vp(flag.data_ptr()), vp(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    assert torch.equal(u, u0.view(P, w.R))
    assert torch.equal(slot, s0.view(E, w.K)) and torch.equal(score, c0.view(E, w.K))
    assert T.dflash2_trace_read(vp(buf.data_ptr()), buf.numel() * 8, 0) == 0
    st = buf.view(512, 64)
    live = st[st[:, 0] > 0]
    assert live.shape[0] > 0
    for a, b in ((0, 1), (1, 4), (4, 31)):
        ok = (live[:, a] > 0) & (live[:, b] > 0)
        assert ok.any() and bool((live[ok, b] >= live[ok, a]).all()), (a, b)
