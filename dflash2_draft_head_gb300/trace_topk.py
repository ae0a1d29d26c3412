"""Row timeline of dflash2_topk's streaming kernel.

Builds libdflash2_trace.so (the top-K kernel compiled with its trace points),
runs dflash2_topk on seeded N(0, 4) logits with L2 flushed before each call,
and prints, for each traced row of the CTAs (their rows 0-3 and 10-13), the
median over CTAs of each point's time after filter warp 0 reached the row, in
microseconds, from the last of `--calls` launches.  Point meanings are listed
with dflash2_trace_read_topk in include/dflash2.h.

    python -m dflash2_draft_head_gb300.trace_topk --rows 4096 --V 151936 --K 16 --dtype bf16
"""
from __future__ import annotations

import argparse
import ctypes

import torch

from . import build as B

POINTS = ["waited for the selector", "first stage done", "filter warp 0 done",
          "selector done", "producer first issue", "producer last issue", "filter warp 7 done"]


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--rows", type=int, default=4096)
    ap.add_argument("--V", type=int, default=151936)
    ap.add_argument("--K", type=int, default=16)
    ap.add_argument("--dtype", choices=["f32", "bf16"], default="f32")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--seed", type=int, default=5)
    a = ap.parse_args()
    lib = ctypes.CDLL(B.build_traced())
    vp = ctypes.c_void_p
    lib.dflash2_trace_read_topk.argtypes = [vp, ctypes.c_int, ctypes.c_int]
    lib.dflash2_topk.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 vp, vp, vp]
    dev = torch.device("cuda", 0)
    g = torch.Generator(device="cpu").manual_seed(a.seed)
    dt = torch.bfloat16 if a.dtype == "bf16" else torch.float32
    x = (torch.randn(a.rows, a.V, generator=g) * 2.0).to(dt).to(dev)
    ids = torch.empty(a.rows, a.K, dtype=torch.int32, device=dev)
    vals = torch.empty(a.rows, a.K, dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    buf = torch.zeros(1024 * 64, dtype=torch.int64)
    for _ in range(max(a.calls, 1)):
        torch.cuda.synchronize()
        if lib.dflash2_trace_read_topk(vp(buf.data_ptr()), buf.numel() * 8, 1) != 0:
            raise RuntimeError("trace read failed")
        flush.zero_()
        if lib.dflash2_topk(vp(x.data_ptr()), a.rows, a.V, a.K, 1 if dt == torch.bfloat16 else 0,
                            vp(ids.data_ptr()), vp(vals.data_ptr()),
                            vp(stream.cuda_stream)) != 0:
            raise RuntimeError(lib.dflash2_last_error().decode())
    torch.cuda.synchronize()
    if lib.dflash2_trace_read_topk(vp(buf.data_ptr()), buf.numel() * 8, 0) != 0:
        raise RuntimeError("trace read failed")
    st = buf.view(1024, 8, 8)
    print(f"{a.rows} x {a.V} {a.dtype}, K = {a.K}: median over CTAs, us after filter warp 0 "
          "reached the row")
    print("  row  " + " | ".join(POINTS))
    for j, r in enumerate((0, 1, 2, 3, 10, 11, 12, 13)):
        b = st[:, j, 0]
        ok = b > 0
        if not ok.any():
            continue
        rel = (st[ok, j, :] - b[ok, None]).float() / 1e3
        rel[st[ok, j, :] == 0] = float("nan")
        meds = [float(rel[:, k].nanmedian()) for k in range(1, 8)]
        nxt = ""
        if j + 1 < 8 and r + 1 == (0, 1, 2, 3, 10, 11, 12, 13)[j + 1]:
            b2 = st[:, j + 1, 0]
            both = ok & (b2 > 0)
            if both.any():
                nxt = f"  (next row +{float((b2[both] - b[both]).float().median()) / 1e3:.2f})"
        print(f"  {r:3d}  " + " | ".join(f"{m:6.2f}" for m in meds) + nxt)


if __name__ == "__main__":
    main()
