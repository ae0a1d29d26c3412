"""The seeded input generator: deterministic, window-consistent, storage-exact (CPU)."""
import torch

from dflash2_draft_head_gb300 import synth
from dflash2_draft_head_gb300.workloads import WORKLOADS, Workload


def _w(**kw):
    base = dict(name="t", S=2, n=9000, C=16, T=4, G=2, d=16, R=8, V=50, K=5, dtype="bf16",
                S_sel=2, n_sel=6, seed=11)
    base.update(kw)
    return Workload(**base)


def test_deterministic():
    w = _w(n=20)
    a = synth.conv_inputs(w)
    b = synth.conv_inputs(w)
    for k in a:
        assert torch.equal(a[k], b[k])


def test_windows_match_full_sequence():
    w = _w()
    full = synth.normal_rows(w.seed, "x", 1, 0, w.n, (w.C,), 1.0, "bf16", w.n)
    for lo, hi in [(0, 10), (4090, 4100), (8000, 9000), (8191, 8193)]:
        part = synth.normal_rows(w.seed, "x", 1, lo, hi, (w.C,), 1.0, "bf16", w.n)
        assert torch.equal(part, full[lo:hi])


def test_bf16_values_are_exact():
    w = _w(n=30)
    x = synth.conv_inputs(w)["x"]
    assert torch.equal(x.to(torch.bfloat16).float(), x)


def test_candidate_ids_distinct_and_in_range():
    w = _w(K=40, V=45, n_sel=50)  # K close to V: exercises the without-replacement draw
    ids = synth.selector_inputs(w)["cand_ids"]
    assert ids.dtype == torch.int32 and ids.shape == (2, 50, 40)
    assert int(ids.min()) >= 0 and int(ids.max()) < 45
    srt, _ = torch.sort(ids, -1)
    assert not (srt[..., 1:] == srt[..., :-1]).any()


def test_distribution_scales():
    w = _w(n=4096, C=64, T=4, G=8, R=64, V=4000, d=256, dtype="f32")
    c = synth.conv_inputs(w)
    cb = synth.codebooks(w)
    assert abs(float(c["x"].std()) - 1.0) < 0.02
    assert abs(float(c["delta"].var()) - 0.1 / 4) < 0.002
    assert abs(float(cb["A"].var()) - 1 / 8) < 0.005          # variance 1/sqrt(R)
    assert abs(float(cb["W"].var()) - 1 / 256) < 0.0005       # variance 1/d


def test_workload_table():
    names = [w.name for w in WORKLOADS]
    assert len(set(names)) == 5
    for w in WORKLOADS:
        assert w.C % w.G == 0 and w.cg % 8 == 0 and w.C % 8 == 0
        assert w.K <= w.V and w.R % 8 == 0
