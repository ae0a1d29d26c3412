"""GPU parity of the CUDA path against the fp64 oracle (needs a GB300).

Every call goes through the C ABI (libdflash2.so) via the thin binding.
Inputs come from the seeded generator; the oracle sees the same (bf16-rounded)
values in double precision.  Covered: the five workloads at full size (the
long-span convolution on sampled windows), small ragged shapes that span
several tiles, and the degenerate cases (n = 1, n < T, T = 1, G = 1, 8
channels per group, no history, K = 1, R not a multiple of 16, ...).
"""
import math

import numpy as np
import pytest
import torch

import dflash2_draft_head_gb300 as df2
import oracle
from dflash2_draft_head_gb300 import synth
from dflash2_draft_head_gb300.workloads import WORKLOADS, Workload
from helpers import assert_argmax, assert_close, dev, host

pytestmark = pytest.mark.gpu

BY = {w.name: w for w in WORKLOADS}


@pytest.fixture(scope="module", autouse=True)
def _built():
    df2.build_library()
    df2.lib()
    yield
    assert df2.take_device_faults() == 0


def W_(name="case", S=2, n=9, C=64, T=4, G=4, d=64, R=16, V=300, K=4, dtype="bf16", S_sel=None,
       n_sel=None, seed=7):
    return Workload(name=name, S=S, n=n, C=C, T=T, G=G, d=d, R=R, V=V, K=K, dtype=dtype,
                    S_sel=S if S_sel is None else S_sel, n_sel=n if n_sel is None else n_sel,
                    seed=seed)


# ------------------------------------------------------------------ dynconv

def check_dynconv(w, out_dtype=None, with_hist=True):
    inp = synth.conv_inputs(w, with_hist=with_hist)
    od = out_dtype or w.dtype
    out = df2.dynconv(dev(inp["x"], w.dtype), dev(inp["hist"], w.dtype), dev(inp["base"], w.dtype),
                      dev(inp["delta"], w.dtype),
                      out_dtype=torch.bfloat16 if od == "bf16" else torch.float32)
    torch.cuda.synchronize()
    ref = oracle.dynconv(inp["x"].numpy(), None if inp["hist"] is None else inp["hist"].numpy(),
                         inp["base"].numpy(), inp["delta"].numpy())
    return assert_close(host(out), ref, w.dtype, f"dynconv {w.name}")


@pytest.mark.parametrize("name", [w.name for w in WORKLOADS if w.name != "longspan_8x32768_T8"])
def test_dynconv_workloads(name):
    check_dynconv(BY[name])


@pytest.mark.parametrize("name", ["qwen27b_single_block16", "batched_256x16_d5120"])
def test_dynconv_workloads_fp32_out(name):
    check_dynconv(BY[name], out_dtype="f32")


@pytest.mark.parametrize("kw", [
    dict(S=3, n=37, C=200, T=5, G=5),      # ragged positions, 25 channel vectors, 40 ch/group
    dict(S=1, n=1, C=64, T=4, G=2),        # one position: all taps but t=0 from history
    dict(S=2, n=3, C=128, T=8, G=4),       # n < T
    dict(S=2, n=11, C=96, T=1, G=3),       # T = 1
    dict(S=2, n=13, C=256, T=16, G=32),    # maximum T, 8 channels per group
    dict(S=1, n=20, C=5376, T=4, G=1),     # one group; C/8 = 672 channel vectors
    dict(S=5, n=17, C=1040, T=3, G=130),   # cg = 8, many groups per block
    dict(S=2, n=40, C=2048, T=12, G=16),   # long taps, tile of 4
    dict(S=3, n=21, C=1024, T=8, G=16),    # 4-position tiles whose halo mixes history and x
    dict(S=1, n=7, C=1024, T=6, G=8),      # T-1 > tile length: halo spans two tiles
])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_dynconv_edge_shapes(kw, dtype):
    check_dynconv(W_(dtype=dtype, **kw))


@pytest.mark.parametrize("kw,hist", [
    (dict(S=100, n=13, C=5120, T=4, G=40), True),   # more tiles than resident CTAs, ragged
    (dict(S=77, n=21, C=5120, T=5, G=40), False),   # ragged tiles, no history
    (dict(S=256, n=16, C=5120, T=2, G=40), True),   # T = 2
    # rows of G bf16 that are whole 128-byte lines: staged delta positions staggered
    (dict(S=3, n=21, C=5120, T=8, G=64), True),     # the long-span shape, ragged tile
    (dict(S=2, n=13, C=1024, T=3, G=128), False),   # cg = 8, no history
    (dict(S=2, n=5, C=512, T=6, G=64), True),       # one partial tile, 64-thread block
])
def test_dynconv_many_tiles(kw, hist):
    """Shapes with more (sequence, tile) items than resident CTAs (bf16 pipelined path)."""
    check_dynconv(W_(dtype="bf16", **kw), with_hist=hist)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("T", [4, 8])
def test_dynconv_null_history(dtype, T):
    check_dynconv(W_(S=3, n=13, C=128, T=T, G=8, dtype=dtype), with_hist=False)


def test_dynconv_block_split_matches_one_run():
    """Running block by block with the carried (T-1)-row history equals one run."""
    w = W_(S=2, n=48, C=512, T=4, G=8)
    inp = synth.conv_inputs(w)
    x = dev(inp["x"], "bf16")
    hist = dev(inp["hist"], "bf16")
    base = dev(inp["base"], "bf16")
    delta = dev(inp["delta"], "bf16")
    full = df2.dynconv(x, hist, base, delta, out_dtype=torch.float32)
    xx = torch.cat([hist, x], 1)
    for i0 in range(0, 48, 16):
        part = df2.dynconv(x[:, i0:i0 + 16].contiguous(), xx[:, i0:i0 + 3].contiguous(), base,
                           delta[:, i0:i0 + 16].contiguous(), out_dtype=torch.float32)
        torch.testing.assert_close(part, full[:, i0:i0 + 16], rtol=0, atol=0)


def test_dynconv_longspan_sampled_windows():
    """8 x 32768 positions, T=8, G=64 at full size; oracle on sampled windows."""
    w = BY["longspan_8x32768_T8"]
    T = w.T
    sd = w.seed
    x_d = torch.empty((w.S, w.n, w.C), dtype=torch.bfloat16, device="cuda")
    windows = {}
    rng = np.random.default_rng(3)
    starts = {s: [0, int(rng.integers(T, w.n - 512)), w.n - 256] for s in range(w.S)}
    for s in range(w.S):
        xs = synth.normal_rows(sd, "x", s, 0, w.n, (w.C,), 1.0, w.dtype, w.n)
        x_d[s].copy_(xs.to(torch.bfloat16))
        for a in starts[s]:
            lo = max(0, a - (T - 1))
            windows[(s, a)] = xs[lo:a + 256].clone()
        del xs
    hist = synth.normal_tensor(sd, "hist", w.S, T - 1, (w.C,), 1.0, w.dtype)
    base = synth.normal_whole(sd, "base", (T, w.C), math.sqrt(1.0 / T), w.dtype)
    delta = synth.normal_tensor(sd, "delta", w.S, w.n, (T, w.G), math.sqrt(0.1 / T), w.dtype)
    out = df2.dynconv(x_d, dev(hist, "bf16"), dev(base, "bf16"), dev(delta, "bf16"))
    torch.cuda.synchronize()
    del x_d
    checked = 0
    for (s, a), rows in windows.items():
        if a == 0:
            xw, hw = rows[:256], hist[s]
        else:
            xw, hw = rows[T - 1:], rows[:T - 1]
        ref = oracle.dynconv(xw[None].numpy(), hw[None].numpy(), base.numpy(),
                             delta[s:s + 1, a:a + 256].numpy())
        assert_close(host(out[s:s + 1, a:a + 256]), ref, "bf16", f"longspan s={s} a={a}")
        checked += ref.size
    assert checked >= 2 ** 17


# ------------------------------------------------------------------ project

def check_project(w):
    cb = synth.codebooks(w)
    sel = synth.selector_inputs(w)
    u = df2.project(dev(sel["h"], w.dtype), dev(cb["W"], w.dtype))
    torch.cuda.synchronize()
    ref = oracle.project(sel["h"].numpy(), cb["W"].numpy())
    return assert_close(host(u), ref, w.dtype, f"project {w.name}")


@pytest.mark.parametrize("name", [w.name for w in WORKLOADS])
def test_project_workloads(name):
    check_project(BY[name])


@pytest.mark.parametrize("kw", [
    dict(S=1, n=1, d=64, R=16),            # P = 1
    dict(S=3, n=43, d=200, R=24),          # P = 129 (two M tiles), ragged K block, R % 16 = 8
    dict(S=1, n=8, d=8, R=8),              # smallest legal shape
    dict(S=4, n=64, d=1032, R=136),        # two N tiles, ragged
    dict(S=2, n=100, d=5120, R=512),       # maximum R
    dict(S=64, n=40, d=5120, R=128),       # 20 M tiles
    dict(S=4, n=64, d=1032, R=160),        # two N tiles (the delta predictor's T*G), split-K
    dict(S=64, n=64, d=5120, R=160),       # two N tiles, 32 M tiles
    dict(S=1, n=16, d=5120, R=152),        # two N tiles, ragged R, one M tile
    dict(S=40, n=500, d=512, R=200),       # 157 M tiles: one 256-column tile, ragged R
    dict(S=20, n=1000, d=256, R=512),      # 157 M tiles x two 256-column tiles
])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_project_edge_shapes(kw, dtype):
    check_project(W_(dtype=dtype, C=64, G=4, **kw))


def check_project_ws(w):
    """The workspace variant: oracle parity and bit-identical to the plain call."""
    cb = synth.codebooks(w)
    sel = synth.selector_inputs(w)
    h = dev(sel["h"], w.dtype)
    W = dev(cb["W"], w.dtype)
    nbytes = df2.project_workspace_bytes(w.P, w.d, w.R)
    ws = torch.full((max(nbytes // 4, 1),), float("nan"), device="cuda")  # contents irrelevant
    u_ws = df2.project(h, W, workspace=ws)
    u = df2.project(h, W)
    torch.cuda.synchronize()
    ref = oracle.project(sel["h"].numpy(), cb["W"].numpy())
    assert_close(host(u_ws), ref, w.dtype, f"project_ws {w.name}")
    assert torch.equal(u_ws, u)


@pytest.mark.parametrize("name", [w.name for w in WORKLOADS])
def test_project_ws_workloads(name):
    check_project_ws(BY[name])


@pytest.mark.parametrize("kw", [
    dict(S=1, n=1, d=64, R=16),
    dict(S=3, n=43, d=200, R=24),
    dict(S=4, n=64, d=1032, R=136),
    dict(S=2, n=100, d=5120, R=512),
    dict(S=64, n=40, d=5120, R=128),
    dict(S=4, n=64, d=1032, R=160),
    dict(S=64, n=64, d=5120, R=160),
    dict(S=1, n=16, d=5120, R=152),
])
def test_project_ws_edge_shapes(kw):
    check_project_ws(W_(C=64, G=4, **kw))


# ------------------------------------------------------------------ edges

def check_edges(w, with_edges=True, u_src=None):
    cb = synth.codebooks(w)
    sel = synth.selector_inputs(w)
    u = oracle.project(sel["h"].numpy(), cb["W"].numpy()).astype(np.float32)
    e_g, slot_g, score_g = df2.edges(dev(sel["cand_ids"]), dev(torch.from_numpy(u)),
                                     dev(cb["A"], w.dtype), dev(cb["B"], w.dtype),
                                     dev(sel["unary"]), edges_out=with_edges)
    torch.cuda.synchronize()
    e_o, slot_o, score_o = oracle.edges(sel["cand_ids"].numpy(), u, cb["A"].numpy(),
                                        cb["B"].numpy(), sel["unary"].numpy())
    if with_edges:
        assert_close(host(e_g), e_o, w.dtype, f"edges {w.name}")
    assert_close(host(score_g), score_o, w.dtype, f"best_score {w.name}")
    return assert_argmax(host(slot_g), e_o, slot_o, w.dtype, f"argmax {w.name}")


@pytest.mark.parametrize("name", [w.name for w in WORKLOADS])
def test_edges_workloads(name):
    check_edges(BY[name])


def test_edges_without_edge_matrix():
    check_edges(BY["batched_256x16_d5120"], with_edges=False)


@pytest.mark.parametrize("kw", [
    dict(S=3, n=7, K=8, R=24, V=500),      # tile path, R % 16 = 8
    dict(S=2, n=5, K=1, R=64, V=50),       # K = 1: the readout is slot 0
    dict(S=5, n=9, K=3, R=16, V=100),      # warp path (K not a power of two)
    dict(S=3, n=6, K=32, R=128, V=4000),   # tile path, 4 transitions per tile
    dict(S=2, n=5, K=128, R=256, V=5000),  # tile path, one transition per tile
    dict(S=2, n=3, K=200, R=64, V=3000),   # warp path, large K
    dict(S=2, n=4, K=16, R=512, V=3000),   # warp path, maximum R
    dict(S=1, n=2, K=64, R=384, V=3000),   # tile path, maximum R
    dict(S=37, n=3, K=16, R=128, V=20000), # ragged last tile (74 transitions)
    # bf16, K a power of two and R in {64, 128, 256}: the selector's edge phase alone
    dict(S=9, n=5, K=4, R=64, V=1000),     # K = 4, R = 64
    dict(S=1300, n=16, K=16, R=128, V=5000),  # 20800 positions: CTAs take two row blocks
])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_edges_edge_shapes(kw, dtype):
    check_edges(W_(dtype=dtype, C=64, G=4, d=64, **kw))


def test_edges_single_position_launches_nothing():
    w = W_(S=2, n=1, K=4, R=16, V=50)
    cb = synth.codebooks(w)
    sel = synth.selector_inputs(w)
    u = torch.zeros((2, 16), device="cuda")
    e, slot, score = df2.edges(dev(sel["cand_ids"]), u, dev(cb["A"], "bf16"),
                               dev(cb["B"], "bf16"), dev(sel["unary"]), edges_out=True)
    assert e.shape == (2, 0, 4, 4) and slot.shape == (2, 0, 4)


@pytest.mark.parametrize("R", [32, 64])  # bf16 R = 64: the selector's edge phase
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_edges_bad_ids_are_clamped_and_flagged(dtype, R):
    w = W_(S=2, n=4, K=8, R=R, V=64, dtype=dtype)
    cb = synth.codebooks(w)
    sel = synth.selector_inputs(w)
    ids = sel["cand_ids"].clone()
    ids[0, 1, 2] = 64      # past the end -> row 63
    ids[1, 2, 5] = -7      # negative -> row 0
    u = oracle.project(sel["h"].numpy(), cb["W"].numpy()).astype(np.float32)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    e_g, slot_g, _ = df2.edges(dev(ids), dev(torch.from_numpy(u)), dev(cb["A"], dtype),
                               dev(cb["B"], dtype), dev(sel["unary"]), edges_out=True,
                               err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) & df2.binding.FLAG_BAD_ID
    clamped = ids.clamp(0, 63)
    e_o, slot_o, _ = oracle.edges(clamped.numpy(), u, cb["A"].numpy(), cb["B"].numpy(),
                                  sel["unary"].numpy())
    assert_close(host(e_g), e_o, dtype, "edges with clamped ids")
    # valid ids leave the flag clear
    flag.zero_()
    df2.edges(dev(sel["cand_ids"]), dev(torch.from_numpy(u)), dev(cb["A"], dtype),
              dev(cb["B"], dtype), dev(sel["unary"]), err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0


# ------------------------------------------------------------------ select

def check_select(w):
    cb = synth.codebooks(w)
    sel = synth.selector_inputs(w)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    u_g, e_g, slot_g, score_g = df2.select(dev(sel["h"], w.dtype), dev(cb["W"], w.dtype),
                                           dev(sel["cand_ids"]), dev(cb["A"], w.dtype),
                                           dev(cb["B"], w.dtype), dev(sel["unary"]),
                                           edges_out=True, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    u_o, e_o, slot_o, score_o = oracle.select(sel["h"].numpy(), cb["W"].numpy(),
                                              sel["cand_ids"].numpy(), cb["A"].numpy(),
                                              cb["B"].numpy(), sel["unary"].numpy())
    assert_close(host(u_g), u_o, w.dtype, f"select u {w.name}")
    assert_close(host(e_g), e_o, w.dtype, f"select edges {w.name}")
    assert_close(host(score_g), score_o, w.dtype, f"select score {w.name}")
    return assert_argmax(host(slot_g), e_o, slot_o, w.dtype, f"select argmax {w.name}")


@pytest.mark.parametrize("name", [w.name for w in WORKLOADS])
def test_select_workloads(name):
    check_select(BY[name])


def test_select_zero_predecessor_codebook_reads_unary():
    """A = 0: every predecessor's readout is argmax(unary) of the next position."""
    w = W_(S=4, n=6, K=16, R=64, V=1000, d=128)
    cb = synth.codebooks(w)
    sel = synth.selector_inputs(w)
    A0 = torch.zeros_like(cb["A"])
    _, e_g, slot_g, score_g = df2.select(dev(sel["h"], "bf16"), dev(cb["W"], "bf16"),
                                         dev(sel["cand_ids"]), dev(A0, "bf16"),
                                         dev(cb["B"], "bf16"), dev(sel["unary"]), edges_out=True)
    torch.cuda.synchronize()
    un = sel["unary"].numpy()
    want = np.broadcast_to(un[:, 1:, None, :], e_g.shape)
    np.testing.assert_array_equal(host(e_g), want)
    np.testing.assert_array_equal(host(slot_g),
                                  np.broadcast_to(np.argmax(un[:, 1:], -1)[..., None],
                                                  slot_g.shape))


# ------------------------------------------------------------------ boundary errors

def test_misaligned_and_aliased_tensors_are_rejected():
    x = torch.zeros((1, 4, 65), dtype=torch.bfloat16, device="cuda")
    xv = x.view(-1)[1:257].view(1, 4, 64)   # 2-byte offset: not 16-byte aligned
    base = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    delta = torch.zeros((1, 4, 4, 8), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(df2.Dflash2Error) as ei:
        df2.dynconv(xv, None, base, delta)
    assert ei.value.status == 1
    xa = torch.zeros((1, 4, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(df2.Dflash2Error) as ei:
        df2.dynconv(xa, None, base, delta, out=xa)
    assert ei.value.status == 1
    with pytest.raises(df2.Dflash2Error) as ei:
        df2.dynconv(torch.zeros((1, 4, 60), dtype=torch.bfloat16, device="cuda"), None,
                    torch.zeros((4, 60), dtype=torch.bfloat16, device="cuda"),
                    torch.zeros((1, 4, 4, 6), dtype=torch.bfloat16, device="cuda"))
    assert ei.value.status == 2
