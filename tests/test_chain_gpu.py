"""GPU parity of the greedy chain readout (p_min cut) against the oracle.

Both sides read the same seeded lattice (unary, edges, the argmax table and
candidate ids drawn on the host; the argmax table is each edge row's numpy
argmax), so the slots, the tokens and the walk must be identical; the shares
p_i agree within fp32 rounding of a softmax (rtol 1e-5), and the cut length
must agree wherever no share lies within that tolerance of p_min.  Also: the
real pipeline (select with edges, then chain) yields a consistent chain.
"""
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


def _lattice(S, n, K, seed, scale=2.0):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, 1 << 20, (S, n, K)).astype(np.int32)
    un = (rng.standard_normal((S, n, K)) * scale).astype(np.float32)
    e = (rng.standard_normal((S, max(n - 1, 0), K, K)) * scale).astype(np.float32)
    bs = e.argmax(axis=-1).astype(np.int32)
    return ids, un, e, bs


def _run(ids, un, e, bs, pm, start=None):
    S, n, K = ids.shape
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    t, p, L = df2.chain(torch.from_numpy(ids).cuda(), torch.from_numpy(un).cuda(),
                        torch.from_numpy(e).cuda() if n > 1 else None,
                        torch.from_numpy(bs).cuda() if n > 1 else None, pm,
                        None if start is None else torch.from_numpy(start).cuda(), flag)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    return t.cpu().numpy(), p.cpu().numpy().astype(np.float64), L.cpu().numpy()


def _check(ids, un, e, bs, pm, start=None):
    t, p, L = _run(ids, un, e, bs, pm, start)
    rt, rp, rL = oracle.chain(ids, un, e if ids.shape[1] > 1 else None,
                              bs if ids.shape[1] > 1 else None, pm, start)
    np.testing.assert_array_equal(t, rt)
    np.testing.assert_allclose(p, rp, rtol=1e-5, atol=1e-7)
    near = np.abs(rp - pm) <= 1e-5 * np.maximum(np.abs(pm), 1e-2)
    for s in range(ids.shape[0]):
        cut = next((i for i in range(ids.shape[1]) if rp[s, i] < pm), ids.shape[1])
        if not near[s, :min(cut + 1, ids.shape[1])].any():
            assert L[s] == rL[s], (s, L[s], rL[s])
        assert L[s] == next((i for i in range(ids.shape[1]) if p[s, i] < pm), ids.shape[1])


@pytest.mark.parametrize("S,n,K", [(5, 1, 4), (3, 2, 1), (7, 9, 16), (4, 16, 64), (2, 16, 256),
                                   (3, 5, 300), (300, 16, 16)])
@pytest.mark.parametrize("pm", [0.0, 0.3, 0.9, 1.5])
def test_chain_parity(S, n, K, pm):
    _check(*_lattice(S, n, K, S * 1000 + n * 10 + K), pm)


def test_chain_given_start_slots():
    ids, un, e, bs = _lattice(6, 8, 16, 5)
    start = np.array([-1, 0, 15, 3, -1, 7], np.int32)
    _check(ids, un, e, bs, 0.2, start)


def test_chain_ties_and_flat_rows():
    S, n, K = 4, 6, 8
    ids, un, e, bs = _lattice(S, n, K, 9)
    un[:, 0, :] = np.round(un[:, 0, :])      # ties in the first argmax: lowest slot
    e[1] = 0.0                                # flat rows: share 1/K, slot 0
    bs = e.argmax(axis=-1).astype(np.int32)
    _check(ids, un, e, bs, 0.0)
    _check(ids, un, e, bs, 1.0 / K + 1e-3)


def test_chain_bad_slot_is_clamped_and_flagged():
    ids, un, e, bs = _lattice(2, 4, 8, 3)
    bs[0, 1, :] = 99
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    t, p, L = df2.chain(torch.from_numpy(ids).cuda(), torch.from_numpy(un).cuda(),
                        torch.from_numpy(e).cuda(), torch.from_numpy(bs).cuda(), 0.5, None, flag)
    torch.cuda.synchronize()
    assert int(flag.item()) & 1
    assert np.all(np.isin(t.cpu().numpy()[0], ids[0].reshape(-1)))


@pytest.mark.parametrize("name", ["qwen27b_single_block16", "batched_256x16_d5120",
                                  "wide_selector_64x8_d5376_K64"])
def test_chain_workload_shapes(name):
    w = BY_NAME[name]
    _check(*_lattice(w.S_sel, w.n_sel, w.K, w.seed), 0.05)


def test_chain_after_select_pipeline():
    """select (edges materialised) then chain: slots follow the GPU's own argmax
    table, shares match a softmax of the GPU's own edge rows, and the cut is the
    leading run of shares >= p_min (properties; no oracle input comes from here)."""
    w = BY_NAME["qwen27b_single_block16"]
    cb = synth.codebooks(w)
    si = synth.selector_inputs(w)
    bf = lambda t: t.to(torch.bfloat16).cuda()
    u, e, slot, score = df2.select(bf(si["h"]), bf(cb["W"]), si["cand_ids"].cuda(), bf(cb["A"]),
                                   bf(cb["B"]), si["unary"].cuda(), edges_out=True)
    t, p, L = df2.chain(si["cand_ids"].cuda(), si["unary"].cuda(), e, slot, 0.05)
    torch.cuda.synchronize()
    e, slot, t, p = e.cpu().numpy(), slot.cpu().numpy(), t.cpu().numpy(), p.cpu().numpy()
    ids, un = si["cand_ids"].numpy(), si["unary"].numpy()
    for s in range(w.S_sel):
        sl = int(np.argmax(un[s, 0]))
        for i in range(w.n_sel):
            if i > 0:
                row = e[s, i - 1, sl].astype(np.float64)
                nxt = int(slot[s, i - 1, sl])
                q = np.exp(row - row.max())
                assert abs(p[s, i] - q[nxt] / q.sum()) < 1e-5
                sl = nxt
            assert t[s, i] == ids[s, i, sl]
        assert L[s] == next((i for i in range(w.n_sel) if p[s, i] < 0.05), w.n_sel)
