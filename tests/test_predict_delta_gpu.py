"""GPU parity of the delta predictor (delta = x . Wc^T, the conv's taps
predicted from its input) and of predicting then convolving, against the
oracle's projection and convolution (same seeded inputs; bf16 tolerance as
for the projection, which rounds delta to bf16 on the way out)."""
import numpy as np
import pytest
import torch

import dflash2_draft_head_gb300 as df2
import oracle
from dflash2_draft_head_gb300 import synth
from dflash2_draft_head_gb300.workloads import BY_NAME, Workload
from helpers import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    df2.build_library()
    df2.lib()
    yield
    assert df2.take_device_faults() == 0


def _w(S, n, C, T, G, dtype, seed):
    return Workload(name="pd", S=S, n=n, C=C, T=T, G=G, d=C, R=16, V=100, K=4, dtype=dtype,
                    S_sel=S, n_sel=n, seed=seed)


def _tdt(dtype):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("S,n,C,T,G", [(1, 3, 64, 4, 2), (2, 37, 256, 4, 8), (3, 50, 512, 8, 8),
                                       (1, 300, 1024, 4, 40), (2, 129, 512, 8, 64)])
def test_predict_delta_parity(S, n, C, T, G, dtype):
    w = _w(S, n, C, T, G, dtype, S * 100 + n)
    x = synth.normal_tensor(w.seed, "x", S, n, (C,), 1.0, dtype)
    Wc = synth.conv_proj(w)
    d = df2.predict_delta(x.to(_tdt(dtype)).cuda(), Wc.to(_tdt(dtype)).cuda(), T, G)
    torch.cuda.synchronize()
    ref = oracle.project(x.reshape(S * n, C).numpy(), Wc.numpy()).reshape(S, n, T, G)
    assert_close(d.float().cpu().numpy(), ref, dtype, f"predict_delta {S}x{n}x{C} T{T} G{G}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_predict_then_convolve(dtype):
    w = _w(2, 40, 512, 4, 8, dtype, 77)
    ci = synth.conv_inputs(w)
    Wc = synth.conv_proj(w)
    t = _tdt(dtype)
    d = df2.predict_delta(ci["x"].to(t).cuda(), Wc.to(t).cuda(), w.T, w.G)
    out = df2.dynconv(ci["x"].to(t).cuda(), ci["hist"].to(t).cuda(), ci["base"].to(t).cuda(), d,
                      out_dtype=torch.float32)
    torch.cuda.synchronize()
    dref = oracle.project(ci["x"].reshape(-1, w.C).numpy(), Wc.numpy()).reshape(2, 40, w.T, w.G)
    ref = oracle.dynconv(ci["x"].numpy(), ci["hist"].numpy(), ci["base"].numpy(), dref)
    assert_close(out.cpu().numpy(), ref, dtype, "predict + dynconv")


@pytest.mark.parametrize("name,S", [("batched_256x16_d5120", 256), ("longspan_8x32768_T8", 1)])
def test_predict_delta_full_size_sampled(name, S):
    """Full-size launch (the long-span shape on one of its 8 sequences: 32768 rows,
    T*G = 512); the oracle computes 64 sampled rows (first, last, random)."""
    w = BY_NAME[name]
    n, C = w.n, w.C
    x = synth.normal_tensor(w.seed, "x", S, n, (C,), 1.0, w.dtype)
    Wc = synth.conv_proj(w)
    d = df2.predict_delta(x.to(torch.bfloat16).cuda(), Wc.to(torch.bfloat16).cuda(), w.T, w.G)
    torch.cuda.synchronize()
    P = S * n
    rows = np.unique(np.concatenate([[0, P - 1], np.random.default_rng(1).integers(0, P, 62)]))
    xf = x.reshape(P, C)[rows].numpy()
    ref = oracle.project(xf, Wc.numpy())
    got = d.reshape(P, w.T * w.G)[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    assert_close(got, ref, "bf16", f"predict_delta {name}")
