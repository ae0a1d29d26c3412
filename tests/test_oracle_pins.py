"""Pins of the fp64 oracle to facts fixed outside it (CPU only).

Each test ties one oracle function to something other than itself: a library
routine (numpy convolve / matmul / argmax), a closed form, an invariant of the
formula in ggml-org/llama.cpp PR #27342 "spec : add DFlash2 support (local
convolution + candidate selector)", Overview, a second brute-force formulation,
or a hand-worked fixture in tests/golden/.  Together they are chosen so that a
dropped term, a wrong sign or index, or a transposed operand fails at least one.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _conv_case(rng, S=2, n=7, C=16, T=3, G=4):
    x = rng.standard_normal((S, n, C))
    hist = rng.standard_normal((S, T - 1, C))
    base = rng.standard_normal((T, C))
    delta = rng.standard_normal((S, n, T, G))
    return x, hist, base, delta


# ---------------------------------------------------------------- dynconv pins

def test_dynconv_golden_hand_worked():
    gold = json.load(open(os.path.join(GOLD, "dynconv_hand.json")))
    for case in gold["cases"]:
        out = oracle.dynconv(np.array(case["x"], float), np.array(case["hist"], float),
                             np.array(case["base"], float), np.array(case["delta"], float))
        np.testing.assert_array_equal(out, np.array(case["out"], float), err_msg=case["name"])


@pytest.mark.parametrize("T", [1, 2, 4, 7])
def test_dynconv_delta_zero_is_numpy_convolve(T):
    """delta = 0 reduces to a static depthwise causal conv: numpy.convolve per channel."""
    rng = _rng(10 + T)
    x, hist, base, delta = _conv_case(rng, S=3, n=9, C=12, T=T, G=3)
    delta[:] = 0.0
    out = oracle.dynconv(x, hist, base, delta)
    S, n, C = x.shape
    for s in range(S):
        for c in range(C):
            seq = np.concatenate([hist[s, :, c], x[s, :, c]])
            ref = np.convolve(seq, base[:, c])[T - 1:T - 1 + n]
            np.testing.assert_allclose(out[s, :, c], ref, rtol=1e-13, atol=1e-13)


def test_dynconv_T1_elementwise():
    """T = 1: out = (base[0,c] + delta[i,0,g(c)]) * x[i,c]."""
    rng = _rng(2)
    S, n, C, G = 2, 5, 12, 4
    x = rng.standard_normal((S, n, C))
    base = rng.standard_normal((1, C))
    delta = rng.standard_normal((S, n, 1, G))
    out = oracle.dynconv(x, None, base, delta)
    gmap = np.arange(C) // (C // G)
    ref = (base[0][None, None, :] + delta[:, :, 0, :][:, :, gmap]) * x
    np.testing.assert_allclose(out, ref, rtol=1e-14, atol=0)


def test_dynconv_linear_in_x_and_hist():
    rng = _rng(3)
    x1, h1, base, delta = _conv_case(rng)
    x2 = rng.standard_normal(x1.shape)
    h2 = rng.standard_normal(h1.shape)
    a, b = 1.75, -0.5
    lhs = oracle.dynconv(a * x1 + b * x2, a * h1 + b * h2, base, delta)
    rhs = a * oracle.dynconv(x1, h1, base, delta) + b * oracle.dynconv(x2, h2, base, delta)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-12, atol=1e-12)


def test_dynconv_group_shares_delta():
    """Adding k to delta[:, :, t, g] equals adding k to base[t, c] for every c of group g."""
    rng = _rng(4)
    x, hist, base, delta = _conv_case(rng, C=16, G=4, T=3)
    cg = 16 // 4
    for t in range(3):
        for g in range(4):
            d2 = delta.copy()
            d2[:, :, t, g] += 0.375
            b2 = base.copy()
            b2[t, g * cg:(g + 1) * cg] += 0.375
            np.testing.assert_allclose(oracle.dynconv(x, hist, base, d2),
                                       oracle.dynconv(x, hist, b2, delta),
                                       rtol=1e-12, atol=1e-12)


def test_dynconv_causal():
    rng = _rng(5)
    x, hist, base, delta = _conv_case(rng, n=9, T=3)
    ref = oracle.dynconv(x, hist, base, delta)
    j = 4
    x2 = x.copy()
    x2[:, j, :] += 1.0
    out = oracle.dynconv(x2, hist, base, delta)
    np.testing.assert_array_equal(out[:, :j], ref[:, :j])
    assert np.all(np.abs(out[:, j:j + 3] - ref[:, j:j + 3]) > 0)
    np.testing.assert_array_equal(out[:, j + 3:], ref[:, j + 3:])
    # history reaches only the first T-1 positions
    h2 = hist + 1.0
    out = oracle.dynconv(x, h2, base, delta)
    np.testing.assert_array_equal(out[:, 2:], ref[:, 2:])
    assert np.all(np.abs(out[:, :2] - ref[:, :2]) > 0)


def test_dynconv_null_hist_is_zero_hist():
    rng = _rng(6)
    x, hist, base, delta = _conv_case(rng)
    np.testing.assert_array_equal(oracle.dynconv(x, None, base, delta),
                                  oracle.dynconv(x, np.zeros_like(hist), base, delta))


@pytest.mark.parametrize("block", [1, 2, 3, 5])
def test_dynconv_block_split_consistency(block):
    """One long run equals consecutive blocks that carry the last T-1 rows as history."""
    rng = _rng(7)
    T = 4
    x, hist, base, delta = _conv_case(rng, S=2, n=11, C=8, T=T, G=2)
    full = oracle.dynconv(x, hist, base, delta)
    xx = np.concatenate([hist, x], axis=1)
    for i0 in range(0, 11, block):
        i1 = min(11, i0 + block)
        part = oracle.dynconv(x[:, i0:i1], xx[:, i0:i0 + T - 1], base, delta[:, i0:i1])
        np.testing.assert_allclose(part, full[:, i0:i1], rtol=0, atol=0)


def test_dynconv_banded_matrix_brute_force():
    """Second formulation: per channel, a banded n x (n+T-1) matrix times [hist; x]."""
    rng = _rng(8)
    S, n, C, T, G = 2, 6, 8, 3, 2
    x, hist, base, delta = _conv_case(rng, S, n, C, T, G)
    out = oracle.dynconv(x, hist, base, delta)
    cg = C // G
    for s in range(S):
        for c in range(C):
            M = np.zeros((n, n + T - 1))
            for i in range(n):
                for t in range(T):
                    M[i, T - 1 + i - t] = base[t, c] + delta[s, i, t, c // cg]
            v = np.concatenate([hist[s, :, c], x[s, :, c]])
            np.testing.assert_allclose(out[s, :, c], M @ v, rtol=1e-13, atol=1e-13)


def test_dynconv_rejects_indivisible_groups():
    with pytest.raises(ValueError):
        oracle.dynconv(np.zeros((1, 2, 6)), None, np.zeros((2, 6)), np.zeros((1, 2, 2, 4)))


# ---------------------------------------------------------------- project pins

def test_project_golden_hand_worked():
    g = json.load(open(os.path.join(GOLD, "selector_hand.json")))["project"]
    np.testing.assert_array_equal(oracle.project(np.array(g["h"], float), np.array(g["W"], float)),
                                  np.array(g["u"], float))


@pytest.mark.parametrize("P,d,R", [(1, 1, 1), (7, 33, 5), (13, 64, 16)])
def test_project_is_numpy_matmul(P, d, R):
    rng = _rng(P * 100 + d)
    h = rng.standard_normal((P, d))
    W = rng.standard_normal((R, d))
    np.testing.assert_allclose(oracle.project(h, W), np.matmul(h, W.T), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- edge pins

def _edge_case(rng, S=2, n=4, K=5, R=6, V=40):
    ids = np.stack([np.stack([rng.choice(V, K, replace=False) for _ in range(n)]) for _ in range(S)])
    u = rng.standard_normal((S * n, R))
    A = rng.standard_normal((V, R))
    B = rng.standard_normal((V, R))
    unary = rng.standard_normal((S, n, K))
    return ids.astype(np.int32), u, A, B, unary


def test_edges_golden_hand_worked():
    g = json.load(open(os.path.join(GOLD, "selector_hand.json")))["edges"]
    e, slot, score = oracle.edges(np.array(g["cand_ids"]), np.array(g["u"], float),
                                  np.array(g["A"], float), np.array(g["B"], float),
                                  np.array(g["unary"], float))
    np.testing.assert_array_equal(e, np.array(g["edges"], float))
    np.testing.assert_array_equal(slot, np.array(g["best_slot"]))
    np.testing.assert_array_equal(score, np.array(g["best_score"], float))


def test_edges_zero_A_gives_unary_and_argmax_unary():
    rng = _rng(20)
    ids, u, A, B, unary = _edge_case(rng)
    e, slot, score = oracle.edges(ids, u, np.zeros_like(A), B, unary)
    S, n, K = ids.shape
    for s in range(S):
        for i in range(1, n):
            for p in range(K):
                np.testing.assert_array_equal(e[s, i - 1, p], unary[s, i])
                assert slot[s, i - 1, p] == np.argmax(unary[s, i])
                assert score[s, i - 1, p] == unary[s, i].max()


def test_edges_R1_closed_form():
    rng = _rng(21)
    ids, u, A, B, unary = _edge_case(rng, R=1)
    e, _, _ = oracle.edges(ids, u, A, B, unary)
    S, n, K = ids.shape
    for s in range(S):
        for i in range(1, n):
            a = A[ids[s, i - 1], 0]
            b = B[ids[s, i], 0]
            ref = np.outer(a * u[s * n + i, 0], b) + unary[s, i][None, :]
            np.testing.assert_allclose(e[s, i - 1], ref, rtol=1e-14, atol=1e-14)


def test_edges_unit_projection_is_bilinear_matmul():
    """u == 1 leaves the plain bilinear form A_P B_C^T + unary (numpy matmul)."""
    rng = _rng(22)
    ids, u, A, B, unary = _edge_case(rng, R=8)
    u[:] = 1.0
    e, _, _ = oracle.edges(ids, u, A, B, unary)
    S, n, K = ids.shape
    for s in range(S):
        for i in range(1, n):
            ref = np.matmul(A[ids[s, i - 1]], B[ids[s, i]].T) + unary[s, i][None, :]
            np.testing.assert_allclose(e[s, i - 1], ref, rtol=1e-13, atol=1e-13)


def test_edges_trilinear():
    rng = _rng(23)
    ids, u, A, B, unary = _edge_case(rng)
    z = np.zeros_like(unary)
    e0, _, _ = oracle.edges(ids, u, A, B, z)
    for which in range(3):
        args = [u, A, B]
        other = rng.standard_normal(args[which].shape)
        a1 = list(args)
        a1[which] = 2.0 * args[which] + other
        a2 = list(args)
        a2[which] = other
        e1, _, _ = oracle.edges(ids, a1[0], a1[1], a1[2], z)
        e2, _, _ = oracle.edges(ids, a2[0], a2[1], a2[2], z)
        np.testing.assert_allclose(e1, 2.0 * e0 + e2, rtol=1e-11, atol=1e-11)


def test_edges_swap_symmetry():
    """(edge - unary) with (A, B) at p->c equals that with (B, A) at c->p."""
    rng = _rng(24)
    V, R, K = 30, 5, 4
    ids0 = rng.choice(V, K, replace=False)
    ids1 = rng.choice(V, K, replace=False)
    u = rng.standard_normal((2, R))
    A = rng.standard_normal((V, R))
    B = rng.standard_normal((V, R))
    z = np.zeros((1, 2, K))
    e, _, _ = oracle.edges(np.array([[ids0, ids1]], np.int32), u, A, B, z)
    e2, _, _ = oracle.edges(np.array([[ids1, ids0]], np.int32), u, B, A, z)
    np.testing.assert_allclose(e[0, 0], e2[0, 0].T, rtol=1e-13, atol=1e-13)


def test_edges_brute_force_einsum_and_argmax():
    rng = _rng(25)
    ids, u, A, B, unary = _edge_case(rng, S=3, n=5, K=6, R=7, V=50)
    e, slot, score = oracle.edges(ids, u, A, B, unary)
    S, n, K = ids.shape
    for s in range(S):
        for i in range(1, n):
            ref = np.einsum("pr,r,cr->pc", A[ids[s, i - 1]], u[s * n + i], B[ids[s, i]]) \
                + unary[s, i][None, :]
            np.testing.assert_allclose(e[s, i - 1], ref, rtol=1e-13, atol=1e-13)
            np.testing.assert_array_equal(slot[s, i - 1], np.argmax(e[s, i - 1], axis=1))
            np.testing.assert_array_equal(score[s, i - 1], e[s, i - 1].max(axis=1))


def test_edges_tie_takes_lowest_slot():
    ids = np.array([[[0, 1, 2], [3, 4, 5]]], np.int32)
    A = np.zeros((6, 2))
    B = np.ones((6, 2))
    u = np.ones((2, 2))
    unary = np.array([[[0, 0, 0], [1.0, 3.0, 3.0]]])
    _, slot, score = oracle.edges(ids, u, A, B, unary)
    np.testing.assert_array_equal(slot[0, 0], [1, 1, 1])
    np.testing.assert_array_equal(score[0, 0], [3.0, 3.0, 3.0])


def test_edges_single_position_has_no_transitions():
    rng = _rng(26)
    ids, u, A, B, unary = _edge_case(rng, n=1)
    e, slot, score = oracle.edges(ids, u, A, B, unary)
    assert e.shape == (2, 0, 5, 5) and slot.shape == (2, 0, 5)


def test_edges_rejects_out_of_range_ids():
    rng = _rng(27)
    ids, u, A, B, unary = _edge_case(rng, V=40)
    ids[1, 2, 3] = 40
    with pytest.raises(ValueError):
        oracle.edges(ids, u, A, B, unary)
    ids[1, 2, 3] = -1
    with pytest.raises(ValueError):
        oracle.edges(ids, u, A, B, unary)


def test_select_is_project_then_edges():
    rng = _rng(28)
    S, n, K, R, V, d = 2, 4, 3, 5, 20, 9
    ids, _, A, B, unary = _edge_case(rng, S, n, K, R, V)
    h = rng.standard_normal((S * n, d))
    W = rng.standard_normal((R, d))
    u, e, slot, score = oracle.select(h, W, ids, A, B, unary)
    np.testing.assert_allclose(u, h @ W.T, rtol=1e-12, atol=1e-12)
    e2, slot2, score2 = oracle.edges(ids, h @ W.T, A, B, unary)
    np.testing.assert_allclose(e, e2, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(slot, slot2)


# ---------------------------------------------------------------- top-K pins

def test_topk_golden_hand_worked():
    g = json.load(open(os.path.join(GOLD, "topk_hand.json")))
    for case in g["cases"]:
        ids, vals = oracle.topk(np.array(case["z"], float), case["K"])
        np.testing.assert_array_equal(ids, np.array(case["ids"]))
        want = np.array(case["vals"], float)
        np.testing.assert_array_equal(vals, want)                # NaN == NaN here
        np.testing.assert_array_equal(np.signbit(vals), np.signbit(want))


@pytest.mark.parametrize("V,K", [(1, 1), (17, 1), (50, 7), (64, 64), (300, 16)])
def test_topk_is_numpy_lexsort(V, K):
    """Library sort: order by (-value, index) and take the first K."""
    rng = _rng(V * 7 + K)
    z = np.round(rng.standard_normal((5, V)) * 4) / 4  # coarse values: many ties
    ids, vals = oracle.topk(z, K)
    for r in range(5):
        order = np.lexsort((np.arange(V), -z[r]))[:K]
        np.testing.assert_array_equal(ids[r], order)
        np.testing.assert_array_equal(vals[r], z[r][order])


def test_topk_k1_is_argmax_and_invariants():
    rng = _rng(31)
    z = rng.standard_normal((8, 1000))
    ids, vals = oracle.topk(z, 1)
    np.testing.assert_array_equal(ids[:, 0], np.argmax(z, axis=1))
    ids, vals = oracle.topk(z, 20)
    assert np.all(np.diff(vals, axis=1) <= 0)                  # non-increasing
    for r in range(8):
        rest = np.delete(z[r], ids[r])
        assert rest.max() <= vals[r].min()                      # nothing better left out
        assert len(set(ids[r].tolist())) == 20


def test_topk_rejects_bad_k():
    with pytest.raises(ValueError):
        oracle.topk(np.zeros((1, 4)), 5)
    with pytest.raises(ValueError):
        oracle.topk(np.zeros((1, 4)), 0)


def test_topk_nan_and_inf_rows():
    """Brute force over a masked row: NaN entries never chosen, -inf only when
    nothing larger is left, short rows padded with id -1."""
    rng = _rng(77)
    z = rng.standard_normal((6, 40))
    z[0, ::3] = np.nan
    z[1, :] = -np.inf
    z[1, 7] = 0.5
    z[2, :] = np.nan
    z[2, 5] = -np.inf
    ids, vals = oracle.topk(z, 30)
    for r in range(6):
        ok = np.flatnonzero(~np.isnan(z[r]))
        order = ok[np.lexsort((ok, -z[r][ok]))][:30]
        m = len(order)
        np.testing.assert_array_equal(ids[r, :m], order)
        np.testing.assert_array_equal(vals[r, :m], z[r][order])
        assert np.all(ids[r, m:] == -1) and np.all(np.isnan(vals[r, m:]))
    assert ids[1, 0] == 7 and ids[1, 1] == 0          # 0.5 first, then -inf by index
    assert ids[2, 0] == 5 and np.all(ids[2, 1:] == -1)


# ---------------------------------------------------------------- chain readout pins

def test_chain_golden_hand_worked():
    g = json.load(open(os.path.join(GOLD, "chain_hand.json")))
    cand = np.array(g["cand_ids"])
    unary = np.log(np.array(g["unary_w"], float))
    edges = np.log(np.array(g["edges_w"], float))
    bs = np.array(g["best_slot"])
    for pm, want_len in g["length"].items():
        t, p, L = oracle.chain(cand, unary, edges, bs, float(pm))
        np.testing.assert_array_equal(t, np.array(g["tokens"]))
        np.testing.assert_allclose(p, np.array(g["probs"]), rtol=1e-12)
        assert int(L[0]) == want_len, pm
    t, p, L = oracle.chain(cand, unary, edges, bs, 0.0, start_slot=np.array([1]))
    np.testing.assert_array_equal(t, np.array(g["start1_tokens"]))
    np.testing.assert_allclose(p, np.array(g["start1_probs"]), rtol=1e-12)


def test_chain_follows_argmax_and_scipy_softmax():
    """Slots from numpy.argmax over the oracle's own edge rows, shares from
    scipy.special.softmax (library routines), on a random lattice."""
    from scipy.special import softmax
    rng = _rng(11)
    S, n, K, R, V = 3, 7, 6, 8, 50
    ids = np.stack([np.stack([rng.choice(V, K, replace=False) for _ in range(n)]) for _ in range(S)])
    u = rng.standard_normal((S * n, R))
    A, B = rng.standard_normal((V, R)), rng.standard_normal((V, R))
    un = rng.standard_normal((S, n, K))
    e, bs, _ = oracle.edges(ids, u, A, B, un)
    t, p, L = oracle.chain(ids, un, e, bs, 0.0)
    for s in range(S):
        slot = int(np.argmax(un[s, 0]))
        assert abs(p[s, 0] - softmax(un[s, 0])[slot]) < 1e-12
        assert t[s, 0] == ids[s, 0, slot]
        for i in range(1, n):
            row = e[s, i - 1, slot]
            nxt = int(np.argmax(row))
            assert abs(p[s, i] - softmax(row)[nxt]) < 1e-12
            slot = nxt
            assert t[s, i] == ids[s, i, slot]
        assert L[s] == n


def test_chain_cut_closed_forms():
    rng = _rng(12)
    S, n, K = 4, 5, 3
    ids = rng.integers(0, 100, (S, n, K)).astype(np.int32)
    un = rng.standard_normal((S, n, K))
    e = rng.standard_normal((S, n - 1, K, K))
    bs = e.argmax(axis=-1).astype(np.int32)
    _, p, L0 = oracle.chain(ids, un, e, bs, 0.0)
    assert np.all(L0 == n) and np.all((p > 0) & (p <= 1))
    _, _, L1 = oracle.chain(ids, un, e, bs, 1.01)
    assert np.all(L1 == 0)
    prev = L0
    for pm in np.linspace(0.0, 1.0, 21):                 # non-increasing in p_min
        _, pp, Lm = oracle.chain(ids, un, e, bs, pm)
        assert np.all(Lm <= prev)
        for s in range(S):                                 # = leading run of p >= p_min
            assert Lm[s] == next((i for i in range(n) if pp[s, i] < pm), n)
        prev = Lm
    # constant rows: every share is 1/K; K = 1: every share is 1
    _, pc, _ = oracle.chain(ids, np.zeros_like(un), np.zeros_like(e), np.zeros_like(bs), 0.0)
    np.testing.assert_allclose(pc, 1.0 / K, rtol=1e-12)
    _, p1, L1k = oracle.chain(ids[:, :, :1], un[:, :, :1], e[:, :, :1, :1],
                              np.zeros((S, n - 1, 1), np.int32), 1.0)
    np.testing.assert_allclose(p1, 1.0)
    np.testing.assert_array_equal(L1k, n)
    # one position: only p0
    t, p, L = oracle.chain(ids[:, :1], un[:, :1], None, None, 0.5)
    assert t.shape == (S, 1) and np.all(L == (p[:, 0] >= 0.5))


def test_chain_rejects_bad_slot():
    ids = np.zeros((1, 2, 2), np.int32)
    with pytest.raises(ValueError):
        oracle.chain(ids, np.zeros((1, 2, 2)), np.zeros((1, 1, 2, 2)), np.array([[[5, 0]]]), 0.0)
    with pytest.raises(ValueError):
        oracle.chain(ids, np.zeros((1, 2, 2)), np.zeros((1, 1, 2, 2)), np.zeros((1, 1, 2)), 0.0,
                     start_slot=np.array([2]))
