"""GPU parity of the top-K candidate extraction against the oracle (needs a GB300).

Selection is exact work, so the bar is bit-exact: the ids must equal the
oracle's and the values must equal the logits at those ids (NaN padding
included, sign of zero included).  Covered: rows misaligned against 16 bytes
(V not a multiple of 4 or 8), rows shorter than one vector, K = 1, K = V,
K = 1024, many and few rows (one CTA per row and clusters splitting a row),
ties, ascending rows (a selection after every stage), constant rows of +0 and
-0, NaN and -inf, both input dtypes; the draft-logit shapes of the workloads
at full size (sampled rows), the review thread's sweep shapes, and the
extraction feeding the selector.
"""
import zlib

import numpy as np
import pytest
import torch

import dflash2_draft_head_gb300 as df2
import oracle
from dflash2_draft_head_gb300 import synth
from dflash2_draft_head_gb300.workloads import BY_NAME

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    df2.build_library()
    df2.lib()
    yield
    assert df2.take_device_faults() == 0


def _to_dev(z, dtype):
    t = torch.as_tensor(np.ascontiguousarray(z), dtype=torch.float32)
    return (t.to(torch.bfloat16) if dtype == "bf16" else t).cuda()


def _check(ids, vals, z, K, rows=None, what=""):
    """Compare GPU outputs (rows `rows` of the whole) with the oracle on z."""
    gi = ids.cpu().numpy()
    gv = vals.cpu().numpy().astype(np.float64)
    if rows is not None:
        gi, gv = gi[rows], gv[rows]
    ri, rv = oracle.topk(z, K)
    bad = np.argwhere(gi != ri)
    assert bad.size == 0, f"{what}: {len(bad)} id mismatches, first {bad[:3].tolist()} " \
                          f"gpu {gi[tuple(bad[0])]} oracle {ri[tuple(bad[0])]}"
    np.testing.assert_array_equal(gv, rv, err_msg=what)
    np.testing.assert_array_equal(np.signbit(gv), np.signbit(rv), err_msg=what + " sign")


def _storage(z, dtype):
    return synth.to_storage(torch.as_tensor(z, dtype=torch.float32), dtype).numpy() \
        .astype(np.float64)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("rows,V,K", [
    (1, 1, 1), (3, 5, 5), (2, 7, 3), (5, 15, 4), (4, 33, 33), (2, 1000, 16), (7, 4099, 64),
    (2, 70001, 1), (3, 70001, 1024), (40, 9999, 16), (300, 5003, 8), (160, 2048, 1024),
    (17, 151937, 16), (5, 151936, 32), (12, 262144, 16), (16, 8, 8), (1, 262144, 1),
    (6, 50021, 40), (3, 151936, 48), (150, 20011, 63),  # K in (32, 64]: two list registers
])
def test_topk_shapes(rows, V, K, dtype):
    z = _storage(np.random.default_rng(rows * 7919 + V + K).standard_normal((rows, V)) * 2, dtype)
    ids, vals = df2.topk(_to_dev(z, dtype), K)
    torch.cuda.synchronize()
    _check(ids, vals, z, K, what=f"{rows}x{V} K={K} {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["ties", "ascending", "descending", "zeros", "nan", "ninf"])
@pytest.mark.parametrize("rows,V,K", [(3, 20011, 16), (200, 3001, 64), (3, 20000, 16), (2, 4096, 32),
                                      (4, 30011, 48)])
def test_topk_degenerate(kind, rows, V, K, dtype):
    rng = np.random.default_rng(zlib.crc32(f"{kind}/{rows}/{V}".encode()))
    if kind == "ties":
        z = np.round(rng.standard_normal((rows, V)) * 2)
    elif kind == "ascending":
        z = np.tile(np.arange(V, dtype=np.float64) * 0.25, (rows, 1))
    elif kind == "descending":
        z = np.tile(-np.arange(V, dtype=np.float64) * 0.25, (rows, 1))
    elif kind == "zeros":
        z = np.zeros((rows, V))
        z[:, 1::3] = -0.0
    elif kind == "nan":
        z = rng.standard_normal((rows, V))
        z[rng.random((rows, V)) < 0.999] = np.nan   # most rows keep fewer than K entries
        z[0, :] = np.nan
    else:
        z = np.full((rows, V), -np.inf)
        z[:, ::97] = rng.standard_normal((rows, len(range(0, V, 97))))
    z = _storage(z, dtype)
    ids, vals = df2.topk(_to_dev(z, dtype), K)
    torch.cuda.synchronize()
    _check(ids, vals, z, K, what=f"{kind} {rows}x{V} K={K} {dtype}")


def _sampled_full(rows, V, K, dtype, seed, n_sample=48):
    z = synth.logits_rows(seed, 0, rows, V, dtype)
    ids, vals = df2.topk(z.to(torch.bfloat16 if dtype == "bf16" else torch.float32).cuda(), K)
    torch.cuda.synchronize()
    pick = np.unique(np.concatenate([[0, rows - 1], np.random.default_rng(seed).integers(
        0, rows, n_sample)]))
    zs = np.concatenate([synth.logits_rows(seed, int(r), int(r) + 1, V, dtype).numpy()
                         for r in pick]).astype(np.float64)
    _check(ids, vals, zs, K, rows=pick, what=f"full {rows}x{V} K={K} {dtype}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("name", ["qwen27b_single_block16", "batched_256x16_d5120",
                                  "wide_selector_64x8_d5376_K64"])
def test_topk_workloads_full_size(name, dtype):
    w = BY_NAME[name]
    _sampled_full(w.P, w.V, w.K, dtype, w.seed)


@pytest.mark.parametrize("rows,V,K", [(2, 200000, 64), (4096, 200000, 64), (64, 200000, 1024),
                                      (1024, 2048, 1024), (8, 248320, 16)])
def test_topk_review_sweep_shapes(rows, V, K):
    """The review thread's microbenchmark grid (fp32 rows up to 200000 wide,
    K = 64 and 1024) and the 248320-entry vocabulary named there."""
    _sampled_full(rows, V, K, "f32", 31 + rows + K)


def test_topk_feeds_selector():
    """cand_ids and unary from the extraction drive the selector; the chained
    GPU result matches the oracle's extraction followed by the oracle's selector."""
    S, n, V, K, R, d = 2, 6, 3000, 8, 16, 64
    rng = np.random.default_rng(5)
    z = _storage(rng.standard_normal((S * n, V)) * 2, "f32")
    ids, vals = df2.topk(_to_dev(z, "f32"), K)
    h = _storage(rng.standard_normal((S * n, d)), "bf16")
    W = _storage(rng.standard_normal((R, d)) / 8, "bf16")
    A = _storage(rng.standard_normal((V, R)) / 2, "bf16")
    B = _storage(rng.standard_normal((V, R)) / 2, "bf16")
    bf = lambda a: torch.as_tensor(a, dtype=torch.float32).to(torch.bfloat16).cuda()
    u, e, slot, score = df2.select(bf(h), bf(W), ids.view(S, n, K), bf(A), bf(B),
                                   vals.view(S, n, K), edges_out=True)
    torch.cuda.synchronize()
    ri, rv = oracle.topk(z, K)
    np.testing.assert_array_equal(ids.cpu().numpy(), ri)
    _, re, rslot, rscore = oracle.select(h, W, ri.reshape(S, n, K), A, B, rv.reshape(S, n, K))
    from helpers import assert_argmax, assert_close
    assert_close(e.cpu().numpy(), re, "bf16", "chained edges")
    assert_argmax(slot.cpu().numpy(), re, rslot, "bf16", "chained argmax")


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_traced_build_matches_and_records_rows(dtype):
    """The streaming top-K built with its trace points returns the same ids and
    values as the normal library, and each traced row's points are ordered."""
    import ctypes
    from dflash2_draft_head_gb300 import build as B
    rows, V, K = 2048, 4099, 16  # 13-14 rows per CTA: rows 10-13 are traced too
    z = _storage(np.random.default_rng(4321).standard_normal((rows, V)) * 2, dtype)
    x = _to_dev(z, dtype)
    ids0, vals0 = df2.topk(x, K)
    T = ctypes.CDLL(B.build_traced())
    vp = ctypes.c_void_p
    T.dflash2_trace_read_topk.argtypes = [vp, ctypes.c_int, ctypes.c_int]
    T.dflash2_topk.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp]
    ids = torch.empty(rows, K, dtype=torch.int32, device="cuda")
    vals = torch.empty(rows, K, dtype=torch.float32, device="cuda")
    buf = torch.zeros(1024 * 64, dtype=torch.int64)
    torch.cuda.synchronize()
    assert T.dflash2_trace_read_topk(vp(buf.data_ptr()), buf.numel() * 8, 1) == 0
    assert T.dflash2_topk(vp(x.data_ptr()), rows, V, K, 1 if dtype == "bf16" else 0,
                          vp(ids.data_ptr()), vp(vals.data_ptr()),
                          vp(torch.cuda.current_stream().cuda_stream)) == 0
    torch.cuda.synchronize()
    assert torch.equal(ids, ids0.view(rows, K))
    assert torch.equal(vals.view(torch.int32), vals0.view(rows, K).view(torch.int32))
    assert T.dflash2_trace_read_topk(vp(buf.data_ptr()), buf.numel() * 8, 0) == 0
    st = buf.view(1024, 8, 8)
    for j in (0, 4):
        r = st[:, j, :]
        live = r[:, 0] > 0
        assert live.any()
        r = r[live]
        for a, b in ((0, 1), (1, 2), (2, 3), (0, 4)):
            assert bool((r[:, b] >= r[:, a]).all()), (j, a, b)
