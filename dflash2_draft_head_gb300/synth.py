"""Seeded synthetic inputs for the DFlash2 draft head.

This module draws random numbers and rounds them to the storage format; it
holds none of the method's arithmetic.  Both the CUDA path and the oracle are
fed from it, so they read identical values.

Distributions (normal laws written N(mean, variance)):
  x, hist, h ~ N(0, 1); base ~ N(0, 1/T); delta ~ N(0, 0.1/T);
  W ~ N(0, 1/d); A, B ~ N(0, 1/sqrt(R)); unary ~ N(0, 1);
  cand_ids: K distinct ids per position, uniform over [0, V);
  draft logits ~ N(0, 4), one generator per row;
  conv_proj Wc [T*G, C] ~ N(0, 0.1/(T*C)) (so the predicted delta has delta's spread).
bf16 workloads draw fp32 and round once to bf16 (round-to-nearest-even); the
returned fp32 arrays hold those exact bf16 values.

Every tensor is generated in independent chunks of CHUNK rows per sequence,
each from its own torch CPU generator keyed by (seed, tensor, sequence, chunk),
so any window of a very long sequence can be regenerated on its own.
"""
from __future__ import annotations

import math

import torch

CHUNK = 4096

_TAG = {"x": 1, "hist": 2, "base": 3, "delta": 4, "h": 5, "W": 6, "A": 7, "B": 8,
        "unary": 9, "cand": 10, "cand_fix": 11,
        "logits": 12, "conv_proj": 13}


def _gen(seed: int, *key: int) -> torch.Generator:
    v = seed & 0xFFFFFFFF
    for k in key:
        v = (v * 1000003 + int(k) + 0x9E3779B9) & ((1 << 62) - 1)
    g = torch.Generator()
    g.manual_seed(v)
    return g


def to_storage(t: torch.Tensor, dtype: str) -> torch.Tensor:
    """Round fp32 values to the storage dtype and return them as fp32."""
    if dtype == "bf16":
        return t.to(torch.bfloat16).to(torch.float32)
    if dtype == "f32":
        return t.to(torch.float32)
    raise ValueError(dtype)


def normal_rows(seed: int, tag: str, s: int, lo: int, hi: int, row_shape, std: float,
                dtype: str, n_total: int) -> torch.Tensor:
    """Rows [lo, hi) of sequence s (of n_total rows) of a normal tensor.

    Chunk ch covers rows [ch*CHUNK, min((ch+1)*CHUNK, n_total)) and is drawn
    whole from its own generator, so a window depends only on n_total.
    """
    row_shape = tuple(row_shape)
    parts = []
    c0 = lo // CHUNK
    c1 = (hi + CHUNK - 1) // CHUNK if hi > lo else c0
    for ch in range(c0, c1):
        g = _gen(seed, _TAG[tag], s, ch)
        rows = min(CHUNK, n_total - ch * CHUNK)
        blk = torch.randn((rows,) + row_shape, generator=g, dtype=torch.float32)
        a = max(lo, ch * CHUNK) - ch * CHUNK
        b = min(hi, (ch + 1) * CHUNK) - ch * CHUNK
        parts.append(blk[a:b])
    if not parts:
        return torch.empty((0,) + row_shape, dtype=torch.float32)
    out = torch.cat(parts, 0) * std
    return to_storage(out, dtype)


def normal_whole(seed: int, tag: str, shape, std: float, dtype: str) -> torch.Tensor:
    """A small normal tensor drawn in one piece (used for base and W)."""
    g = _gen(seed, _TAG[tag], 0, 0)
    return to_storage(torch.randn(tuple(shape), generator=g, dtype=torch.float32) * std, dtype)


def normal_tensor(seed: int, tag: str, S: int, n: int, row_shape, std: float,
                  dtype: str) -> torch.Tensor:
    """A [S, n, *row_shape] normal tensor (sequence by sequence, chunked)."""
    return torch.stack([normal_rows(seed, tag, s, 0, n, row_shape, std, dtype, n)
                        for s in range(S)], 0) if S > 0 else \
        torch.empty((0, n) + tuple(row_shape))


def cand_rows(seed: int, s: int, lo: int, hi: int, K: int, V: int,
              n_total: int) -> torch.Tensor:
    """Candidate ids of positions [lo, hi) of sequence s: K distinct ids per row."""
    if K > V:
        raise ValueError("K distinct ids need K <= V")
    parts = []
    c0 = lo // CHUNK
    c1 = (hi + CHUNK - 1) // CHUNK if hi > lo else c0
    for ch in range(c0, c1):
        g = _gen(seed, _TAG["cand"], s, ch)
        rows_n = min(CHUNK, n_total - ch * CHUNK)
        ids = torch.randint(0, V, (rows_n, K), generator=g, dtype=torch.int64)
        gfix = _gen(seed, _TAG["cand_fix"], s, ch)
        for attempt in range(9):
            srt, _ = torch.sort(ids, dim=1)
            dup = (srt[:, 1:] == srt[:, :-1]).any(dim=1) if K > 1 else \
                torch.zeros(rows_n, dtype=torch.bool)
            rows = torch.nonzero(dup).flatten()
            if rows.numel() == 0:
                break
            if attempt < 8:
                ids[rows] = torch.randint(0, V, (rows.numel(), K), generator=gfix,
                                          dtype=torch.int64)
            else:  # K close to V: draw the remaining rows without replacement
                for r in rows.tolist():
                    ids[r] = torch.randperm(V, generator=gfix)[:K]
        a = max(lo, ch * CHUNK) - ch * CHUNK
        b = min(hi, (ch + 1) * CHUNK) - ch * CHUNK
        parts.append(ids[a:b])
    if not parts:
        return torch.empty((0, K), dtype=torch.int32)
    return torch.cat(parts, 0).to(torch.int32)


def conv_inputs(w, with_hist: bool = True) -> dict:
    """x [S,n,C], hist [S,T-1,C] (or None), base [T,C], delta [S,n,T,G] (fp32 tensors)."""
    sd = w.seed
    x = normal_tensor(sd, "x", w.S, w.n, (w.C,), 1.0, w.dtype)
    hist = normal_tensor(sd, "hist", w.S, w.T - 1, (w.C,), 1.0, w.dtype) if with_hist else None
    base = normal_whole(sd, "base", (w.T, w.C), math.sqrt(1.0 / w.T), w.dtype)
    delta = normal_tensor(sd, "delta", w.S, w.n, (w.T, w.G), math.sqrt(0.1 / w.T), w.dtype)
    return {"x": x, "hist": hist, "base": base, "delta": delta}


def codebooks(w) -> dict:
    """A, B [V,R] and W [R,d] (fp32 tensors holding storage-dtype values)."""
    sd = w.seed
    std_ab = (1.0 / math.sqrt(w.R)) ** 0.5
    A = normal_rows(sd, "A", 0, 0, w.V, (w.R,), std_ab, w.dtype, w.V)
    B = normal_rows(sd, "B", 0, 0, w.V, (w.R,), std_ab, w.dtype, w.V)
    W = normal_whole(sd, "W", (w.R, w.d), math.sqrt(1.0 / w.d), w.dtype)
    return {"A": A, "B": B, "W": W}


def selector_inputs(w) -> dict:
    """h [S_sel*n_sel, d], cand_ids [S_sel,n_sel,K] int32, unary [S_sel,n_sel,K]."""
    sd = w.seed
    h = normal_tensor(sd, "h", w.S_sel, w.n_sel, (w.d,), 1.0, w.dtype).reshape(w.P, w.d)
    cand = torch.stack([cand_rows(sd, s, 0, w.n_sel, w.K, w.V, w.n_sel) for s in range(w.S_sel)], 0)
    unary = normal_tensor(sd, "unary", w.S_sel, w.n_sel, (w.K,), 1.0, "f32")
    return {"h": h, "cand_ids": cand, "unary": unary}


def logits_rows(seed: int, lo: int, hi: int, V: int, dtype: str, std: float = 2.0) -> torch.Tensor:
    """Rows [lo, hi) of a [rows, V] draft-logit matrix; row r comes from its own
    generator, so any row can be regenerated alone."""
    out = torch.empty((max(hi - lo, 0), V), dtype=torch.float32)
    for r in range(lo, hi):
        g = _gen(seed, _TAG["logits"], r, 0)
        out[r - lo] = torch.randn((V,), generator=g, dtype=torch.float32) * std
    return to_storage(out, dtype)


def conv_proj(w) -> torch.Tensor:
    """Wc [T*G, C] of the delta predictor (fp32 tensor holding storage-dtype values)."""
    return normal_whole(w.seed, "conv_proj", (w.T * w.G, w.C), math.sqrt(0.1 / (w.T * w.C)),
                        w.dtype)
