"""The allocation-free projection entry point, dflash2_project_noalloc.

Some callers cannot allocate device memory (a plugin inside an inference
runtime that owns the device pool, a decode loop where an allocation call may
not run).  For them the library carries its own fixed split-K workspace.  This
test calls that entry point through the C ABI, twice in a row on different
inputs (the shared workspace keeps the previous call's contents), and checks
it against dflash2_project within the bf16 test tolerance, and against the
fp64 oracle on a split-K shape and on a shape whose 256-column tiles need no
workspace at all.  It also checks that shapes needing more than the fixed
workspace are refused cleanly.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import dflash2_draft_head_gb300 as df2
import oracle
from helpers import assert_close

pytestmark = pytest.mark.gpu

FIXED_BYTES = 8 << 20


@pytest.fixture(scope="module")
def L():
    df2.build_library()
    return df2.lib()


def _inputs(P, d, R, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    h = torch.randn(P, d, device="cuda", generator=g).to(torch.bfloat16)
    W = (torch.randn(R, d, device="cuda", generator=g) / d ** 0.5).to(torch.bfloat16)
    return h, W


def _call(fn, h, W, u):
    P, d = h.shape
    R = W.shape[0]
    vp = ctypes.c_void_p
    return fn(vp(h.data_ptr()), vp(W.data_ptr()), vp(u.data_ptr()), P, d, R, 1,
              vp(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("P,d,R", [(16, 5120, 128),     # one draft block: split-K 8
                                   (16, 5120, 160),     # two N tiles: split-K 8
                                   (512, 5376, 256),    # wide selector
                                   (4096, 5120, 128)])  # batched: 8 MiB of workspace
def test_noalloc_matches_project_twice(L, P, d, R):
    assert L.dflash2_project_workspace_bytes(P, d, R) <= FIXED_BYTES
    for seed in (1, 2):  # second call sees the first call's workspace contents
        h, W = _inputs(P, d, R, seed)
        u_ref = torch.empty(P, R, device="cuda")
        u_na = torch.full((P, R), float("nan"), device="cuda")
        assert _call(L.dflash2_project, h, W, u_ref) == 0
        assert _call(L.dflash2_project_noalloc, h, W, u_na) == 0, L.dflash2_last_error()
        torch.cuda.synchronize()
        assert_close(u_na.cpu().numpy(), u_ref.cpu().numpy().astype(np.float64), "bf16",
                     f"noalloc P={P} seed={seed}")
    assert df2.take_device_faults() == 0


def test_noalloc_refuses_oversized_shapes(L):
    d, R = 5120, 128
    P = next(p for p in range(128, 1 << 16, 128)
             if L.dflash2_project_workspace_bytes(p, d, R) > FIXED_BYTES)
    h, W = _inputs(P, d, R, 3)
    u = torch.zeros(P, R, device="cuda")
    assert _call(L.dflash2_project_noalloc, h, W, u) == 2  # DF2_ERR_UNSUPPORTED
    assert b"workspace" in L.dflash2_last_error()
    torch.cuda.synchronize()
    assert float(u.abs().max()) == 0.0  # nothing was launched


def _host(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("shape", ["split", "wide256"])
def test_noalloc_matches_oracle(L, shape):
    if shape == "split":  # one draft block: split-K over a cluster, workspace in use
        P, d, R = 16, 5120, 128
        assert L.dflash2_project_workspace_bytes(P, d, R) > 0
    else:  # one 128-row tile per SM, R > 128: 256-column tiles, no split, no workspace
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        P, d, R = 128 * sms, 512, 256
        assert L.dflash2_project_workspace_bytes(P, d, R) == 0
    for seed in (5, 6):
        h, W = _inputs(P, d, R, seed)
        u = torch.full((P, R), float("nan"), device="cuda")
        assert _call(L.dflash2_project_noalloc, h, W, u) == 0, L.dflash2_last_error()
        torch.cuda.synchronize()
        if P <= 64:
            rows = np.arange(P)
        else:
            rnd = np.random.default_rng(seed).integers(0, P, 256)
            rows = np.unique(np.r_[0:8, P - 8:P, rnd])
        ref = oracle.project(_host(h)[rows], _host(W))
        assert_close(u.cpu().numpy()[rows], ref, "bf16", f"noalloc {shape} seed={seed}")
    assert df2.take_device_faults() == 0
