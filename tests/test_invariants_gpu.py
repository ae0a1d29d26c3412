"""GPU invariants: the CUDA path checked directly against closed forms and
library routines (numpy), not only against the oracle.  fp32 mode (no TF32,
fp32 accumulation) with fp32 tolerances unless stated."""
import numpy as np
import pytest
import torch

import dflash2_draft_head_gb300 as df2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    df2.build_library()
    df2.lib()
    yield
    assert df2.take_device_faults() == 0


def _c(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _conv(x, hist, base, delta):
    out = df2.dynconv(_c(x), None if hist is None else _c(hist), _c(base), _c(delta),
                      out_dtype=torch.float32)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def test_dynconv_zero_delta_is_numpy_convolve():
    """delta = 0: each channel is a causal FIR with taps base[:, c] over [hist; x]."""
    rng = np.random.default_rng(1)
    S, n, C, T, G = 2, 23, 64, 4, 8
    x = rng.standard_normal((S, n, C))
    hist = rng.standard_normal((S, T - 1, C))
    base = rng.standard_normal((T, C))
    out = _conv(x, hist, base, np.zeros((S, n, T, G)))
    for s in range(S):
        full = np.concatenate([hist[s], x[s]], 0).astype(np.float32).astype(np.float64)
        for c in range(C):
            ref = np.convolve(full[:, c], base[:, c].astype(np.float32))[T - 1:T - 1 + n]
            np.testing.assert_allclose(out[s, :, c], ref, rtol=1e-5, atol=1e-5)


def test_dynconv_single_tap_is_elementwise():
    rng = np.random.default_rng(2)
    S, n, C, G = 3, 17, 128, 16
    x, base = rng.standard_normal((S, n, C)), rng.standard_normal((1, C))
    delta = rng.standard_normal((S, n, 1, G))
    out = _conv(x, None, base, delta)
    g = np.arange(C) // (C // G)
    f = lambda a: a.astype(np.float32).astype(np.float64)
    ref = (f(base)[0][None, None, :] + f(delta)[:, :, 0, g]) * f(x)
    np.testing.assert_allclose(out, ref, rtol=1e-5, atol=1e-5)


def test_dynconv_is_linear_in_x_and_hist():
    rng = np.random.default_rng(3)
    S, n, C, T, G = 2, 19, 64, 4, 8
    x1, x2 = rng.standard_normal((2, S, n, C)).astype(np.float32)
    h1, h2 = rng.standard_normal((2, S, T - 1, C)).astype(np.float32)
    base = rng.standard_normal((T, C)).astype(np.float32)
    delta = (0.3 * rng.standard_normal((S, n, T, G))).astype(np.float32)
    lhs = _conv(x1 + 0.5 * x2, h1 + 0.5 * h2, base, delta)
    rhs = _conv(x1, h1, base, delta) + 0.5 * _conv(x2, h2, base, delta)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-4, atol=1e-4)


def _edges_f32(ids, u, A, B, unary):
    e, slot, score = df2.edges(torch.from_numpy(ids.astype(np.int32)).cuda(), _c(u), _c(A), _c(B),
                               _c(unary), edges_out=True)
    torch.cuda.synchronize()
    return e.cpu().numpy().astype(np.float64), slot.cpu().numpy(), score.cpu().numpy()


def test_edges_rank_one_closed_form():
    """R = 1 is not a supported rank (R % 8), so R = 8 with one live column."""
    rng = np.random.default_rng(4)
    S, n, K, R, V = 2, 6, 8, 8, 40
    ids = np.stack([np.stack([rng.choice(V, K, replace=False) for _ in range(n)]) for _ in range(S)])
    A, B = np.zeros((V, R)), np.zeros((V, R))
    a, b = rng.standard_normal(V), rng.standard_normal(V)
    A[:, 3], B[:, 3] = a, b
    u = rng.standard_normal((S * n, R))
    unary = rng.standard_normal((S, n, K))
    e, slot, score = _edges_f32(ids, u, A, B, unary)
    f = lambda v: v.astype(np.float32).astype(np.float64)
    for s in range(S):
        for i in range(1, n):
            ref = (f(a)[ids[s, i - 1]][:, None] * f(u)[s * n + i, 3] * f(b)[ids[s, i]][None, :]
                   + f(unary)[s, i][None, :])
            np.testing.assert_allclose(e[s, i - 1], ref, rtol=1e-5, atol=1e-5)
            np.testing.assert_array_equal(slot[s, i - 1], np.argmax(e[s, i - 1], axis=1))


def test_edges_unit_u_is_a_bilinear_form():
    """u = 1: e = A[ids_prev] B[ids]^T + unary (numpy matmul)."""
    rng = np.random.default_rng(5)
    S, n, K, R, V = 2, 5, 16, 32, 100
    ids = np.stack([np.stack([rng.choice(V, K, replace=False) for _ in range(n)]) for _ in range(S)])
    A, B = rng.standard_normal((V, R)), rng.standard_normal((V, R))
    u = np.ones((S * n, R))
    unary = rng.standard_normal((S, n, K))
    e, _, _ = _edges_f32(ids, u, A, B, unary)
    f = lambda v: v.astype(np.float32).astype(np.float64)
    for s in range(S):
        for i in range(1, n):
            ref = f(A)[ids[s, i - 1]] @ f(B)[ids[s, i]].T + f(unary)[s, i][None, :]
            np.testing.assert_allclose(e[s, i - 1], ref, rtol=1e-5, atol=1e-4)


def test_topk_k1_is_numpy_argmax_and_ascending_rows():
    rng = np.random.default_rng(6)
    z = rng.standard_normal((33, 20011)).astype(np.float32)
    ids, vals = df2.topk(_c(z), 1)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids.cpu().numpy()[:, 0], np.argmax(z, axis=1))
    asc = np.tile(np.arange(5000, dtype=np.float32), (3, 1))
    ids, vals = df2.topk(_c(asc), 10)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(ids.cpu().numpy(), np.tile(np.arange(4999, 4989, -1), (3, 1)))
