"""GPU parity of the fused conv with predicted taps (delta = x . Wc^T computed
and used inside one kernel) against the oracle's projection followed by its
convolution, on the same seeded inputs.  Tolerance: the bf16 one of the
projection and the conv (delta is rounded to bf16 between the two steps, as
the unfused pair stores it)."""
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


def _w(S, n, C, T, G, seed):
    return Workload(name="dp", S=S, n=n, C=C, T=T, G=G, d=C, R=16, V=100, K=4, dtype="bf16",
                    S_sel=S, n_sel=n, seed=seed)


def _run(w, with_hist=True, out_dtype=torch.float32, seqs=None):
    ci = synth.conv_inputs(w, with_hist=with_hist)
    Wc = synth.conv_proj(w)
    b = torch.bfloat16
    hist = ci["hist"].to(b).cuda() if with_hist else None
    out = df2.dynconv_predicted(ci["x"].to(b).cuda(), hist, ci["base"].to(b).cuda(),
                                Wc.to(b).cuda(), w.G, out_dtype=out_dtype)
    torch.cuda.synchronize()
    sel = slice(None) if seqs is None else torch.as_tensor(seqs)
    x = ci["x"][sel].numpy()
    S = x.shape[0]
    dref = oracle.project(x.reshape(S * w.n, w.C), Wc.numpy()).reshape(S, w.n, w.T, w.G)
    h = ci["hist"][sel].numpy() if with_hist else None
    ref = oracle.dynconv(x, h, ci["base"].numpy(), dref)
    got = out[sel.cuda() if seqs is not None else sel].float().cpu().numpy()
    return got, ref


# (S, n, C, T, G): one 64-channel block (cluster of 1); clusters of 2, 4 and 8;
# T*G = 168 and 200 (MMA N padded to 176 / 208); a ragged last channel block
# (C = 200); channel slices that split a group (C = 5376 over 8 CTAs); T = 1..8;
# strips that cross sequence boundaries (n = 37, 50, 129); n = 1.
CASES = [
    (1, 3, 64, 4, 4),
    (2, 37, 512, 4, 8),
    (3, 50, 1024, 8, 16),
    (1, 300, 1280, 4, 40),
    (2, 129, 512, 8, 32),
    (1, 20, 5376, 4, 42),
    (1, 40, 200, 8, 25),
    (2, 9, 128, 1, 16),
    (2, 17, 256, 3, 8),
    (3, 11, 384, 2, 12),
    (2, 13, 640, 5, 16),
    (1, 70, 768, 6, 4),
    (2, 21, 448, 7, 8),
    (40, 1, 256, 4, 8),
]


@pytest.mark.parametrize("S,n,C,T,G", CASES)
def test_fused_parity(S, n, C, T, G):
    w = _w(S, n, C, T, G, 1000 + S * 37 + n * 11 + C + T)
    got, ref = _run(w)
    assert_close(got, ref, "bf16", f"dynconv_predicted {S}x{n}x{C} T{T} G{G}")


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_fused_without_history_and_out_dtypes(out_dtype):
    w = _w(2, 37, 512, 4, 8, 4242)
    got, ref = _run(w, with_hist=False, out_dtype=out_dtype)
    assert_close(got, ref, "bf16", f"dynconv_predicted no-hist {out_dtype}")


def test_fused_more_tiles_than_sms():
    # 25600 positions: 200 tiles of 128, each its own CTA (cluster of 1), in two waves
    w = _w(64, 400, 256, 4, 8, 777)
    got, ref = _run(w)
    assert_close(got, ref, "bf16", "dynconv_predicted 64x400x256")


@pytest.mark.parametrize("name,seqs", [
    ("batched_256x16_d5120", [0, 1, 100, 255]),
    ("qwen27b_single_block16", None),
    ("wide_selector_64x8_d5376_K64", [0, 17, 63]),
])
def test_fused_full_size(name, seqs):
    """The full workload in one launch; the oracle computes the listed
    sequences (independent of one another) or all of them."""
    w = BY_NAME[name]
    got, ref = _run(w, seqs=seqs)
    assert_close(got, ref, "bf16", f"dynconv_predicted {name}")


def test_fused_matches_predict_then_convolve():
    """The fused call and the unfused pair it replaces, on the same device
    inputs (they differ only where the split-K order moves a delta across a
    bf16 rounding boundary)."""
    w = _w(4, 100, 1024, 4, 32, 99)
    ci = synth.conv_inputs(w)
    Wc = synth.conv_proj(w)
    b = torch.bfloat16
    x, hist, base = (ci[k].to(b).cuda() for k in ("x", "hist", "base"))
    Wd = Wc.to(b).cuda()
    fused = df2.dynconv_predicted(x, hist, base, Wd, w.G, out_dtype=torch.float32)
    pair = df2.dynconv(x, hist, base, df2.predict_delta(x, Wd, w.T, w.G), out_dtype=torch.float32)
    torch.cuda.synchronize()
    f = fused.cpu().numpy()
    p = pair.cpu().numpy()
    assert_close(f, p, "bf16", "fused vs pair")


def _wf(S, n, C, T, G, seed):
    return Workload(name="dpf", S=S, n=n, C=C, T=T, G=G, d=C, R=16, V=100, K=4, dtype="f32",
                    S_sel=S, n_sel=n, seed=seed)


@pytest.mark.parametrize("S,n,C,T,G,hist", [
    (1, 8, 256, 4, 8, True),      # the tiny all-fp32 workload's shape
    (2, 37, 512, 4, 8, True),
    (3, 50, 200, 8, 25, True),
    (2, 9, 128, 1, 16, True),
    (40, 1, 256, 4, 8, False),
    (3, 21, 384, 3, 8, False),
])
def test_fused_fp32_parity(S, n, C, T, G, hist):
    """All-fp32 mode: delta in exact fp32 (no rounding between the steps)."""
    w = _wf(S, n, C, T, G, 500 + S + n + C + T)
    ci = synth.conv_inputs(w, with_hist=hist)
    Wc = synth.conv_proj(w)
    out = df2.dynconv_predicted(ci["x"].cuda(), ci["hist"].cuda() if hist else None,
                                ci["base"].cuda(), Wc.cuda(), w.G)
    torch.cuda.synchronize()
    assert out.dtype == torch.float32
    dref = oracle.project(ci["x"].reshape(-1, C).numpy(), Wc.numpy()).reshape(S, n, T, G)
    ref = oracle.dynconv(ci["x"].numpy(), ci["hist"].numpy() if hist else None,
                         ci["base"].numpy(), dref)
    assert_close(out.cpu().numpy(), ref, "f32", f"dynconv_predicted fp32 {S}x{n}x{C} T{T}")


def test_fused_rejects_fp32_to_bf16_and_wide_taps():
    w = _wf(1, 8, 128, 4, 8, 5)
    ci = synth.conv_inputs(w)
    Wc = synth.conv_proj(w)
    x = ci["x"].cuda()
    with pytest.raises(df2.Dflash2Error):
        df2.dynconv_predicted(x, ci["hist"].cuda(), ci["base"].cuda(), Wc.cuda(), w.G,
                              out_dtype=torch.bfloat16)
    b = torch.bfloat16
    xb = torch.zeros((1, 8, 2048), dtype=b, device="cuda")
    with pytest.raises(df2.Dflash2Error):  # T*G = 512
        df2.dynconv_predicted(xb, None, torch.zeros((8, 2048), dtype=b, device="cuda"),
                              torch.zeros((512, 2048), dtype=b, device="cuda"), 64)
