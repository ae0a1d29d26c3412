"""Synthetic DFlash2 draft-head workloads (shapes and dtypes only, no arithmetic).

Shapes follow the decode regime the DFlash2 pull request (ggml-org/llama.cpp
#27342, "spec : add DFlash2 support (local convolution + candidate selector)")
runs: draft blocks of 8 or 16 positions over Qwen-27B-shaped hidden states
(d = 5120) and a Gemma-31B-shaped variant (d = 5376), with the materialised
vocab-indexed codebooks its review discusses.  Real checkpoints, prompts and
datasets are not used; every tensor is seeded and synthetic.
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    S: int          # sequences (convolution)
    n: int          # positions per sequence (convolution)
    C: int          # channels
    T: int          # taps
    G: int          # delta groups
    d: int          # hidden size fed to project(h)
    R: int          # codebook rank
    V: int          # vocabulary rows of each codebook
    K: int          # candidates per position
    dtype: str      # "f32" (everything fp32) or "bf16" (bf16 in, fp32 accumulate)
    S_sel: int      # sequences (selector)
    n_sel: int      # positions per sequence (selector)
    seed: int

    @property
    def cg(self) -> int:
        return self.C // self.G

    @property
    def P(self) -> int:
        return self.S_sel * self.n_sel

    @property
    def E(self) -> int:
        return self.S_sel * max(self.n_sel - 1, 0)

    @property
    def out_dtype(self) -> str:
        return self.dtype


def _w(name, S, n, C, T, G, R, V, K, dtype, S_sel=None, n_sel=None, d=None, idx=0):
    return Workload(name=name, S=S, n=n, C=C, T=T, G=G, d=C if d is None else d, R=R, V=V,
                    K=K, dtype=dtype, S_sel=S if S_sel is None else S_sel,
                    n_sel=n if n_sel is None else n_sel, seed=20260 + idx)


# The five workloads, in order: a tiny all-fp32 case, one Qwen-27B-shaped draft
# step, the batched verification regime (the benchmark workload), the long-span
# convolution, and the wide selector.
WORKLOADS = [
    _w("tiny_fp32", 1, 8, 256, 4, 8, 16, 1000, 4, "f32", idx=0),
    _w("qwen27b_single_block16", 1, 16, 5120, 4, 40, 128, 151936, 16, "bf16", idx=1),
    _w("batched_256x16_d5120", 256, 16, 5120, 4, 40, 128, 151936, 16, "bf16", idx=2),
    _w("longspan_8x32768_T8", 8, 32768, 5120, 8, 64, 128, 151936, 16, "bf16",
       S_sel=8, n_sel=16, idx=3),
    _w("wide_selector_64x8_d5376_K64", 64, 8, 5376, 4, 42, 256, 262144, 64, "bf16", idx=4),
]

BY_NAME = {w.name: w for w in WORKLOADS}
BENCH_WORKLOAD = WORKLOADS[2]
