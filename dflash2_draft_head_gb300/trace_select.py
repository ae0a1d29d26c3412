"""Phase timeline of dflash2_select's one-kernel path on a named workload.

Builds libdflash2_trace.so (the selector compiled with its trace points), runs
the selector on the workload's seeded synthetic inputs with L2 flushed before
each call, and prints, for every trace point, the median over the CTAs that
reached it of (stamp - the earliest CTA's entry stamp) in microseconds, from
the last of `--calls` launches.  Slot meanings are listed with
dflash2_trace_read in include/dflash2.h.

    python -m dflash2_draft_head_gb300.trace_select batched_256x16_d5120
"""
from __future__ import annotations

import argparse
import ctypes
import json

import torch

from . import build as B
from . import synth
from .workloads import BY_NAME

SLOTS = {0: "entry, set-up done", 1: "previous grid complete", 2: "first TMA stage landed",
         3: "last projection MMAs committed", 4: "accumulators complete",
         5: "cluster barrier passed", 6: "partials received", 7: "u slice written",
         8: "every edge unit's gathers issued", 31: "CTA exit"}
for _j in range(6):
    SLOTS[9 + _j] = f"edge unit {_j} issued"
    SLOTS[15 + _j] = f"edge unit {_j} landed"
    SLOTS[21 + _j] = f"edge unit {_j} MMAs committed"
for _j in range(4):
    SLOTS[27 + _j] = f"edge unit {_j} scored"


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("workload", nargs="?", default="batched_256x16_d5120")
    ap.add_argument("--calls", type=int, default=5)
    ap.add_argument("--json", action="store_true")
    a = ap.parse_args()
    lib = ctypes.CDLL(B.build_traced())
    vp = ctypes.c_void_p
    lib.dflash2_trace_read.argtypes = [vp, ctypes.c_int, ctypes.c_int]
    w = BY_NAME[a.workload]
    dev = torch.device("cuda", 0)
    cb = synth.codebooks(w)
    si = synth.selector_inputs(w)
    bt = torch.bfloat16
    h, W, A, Bm = (t.to(bt).to(dev) for t in (si["h"], cb["W"], cb["A"], cb["B"]))
    ids, un = si["cand_ids"].to(dev), si["unary"].to(dev)
    P, E = w.S_sel * w.n_sel, w.S_sel * (w.n_sel - 1)
    u = torch.empty((P, w.R), dtype=torch.float32, device=dev)
    slot = torch.empty((E, w.K), dtype=torch.int32, device=dev)
    score = torch.empty((E, w.K), dtype=torch.float32, device=dev)
    flag = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    args = (vp(h.data_ptr()), vp(W.data_ptr()), vp(ids.data_ptr()), vp(A.data_ptr()),
            vp(Bm.data_ptr()), vp(un.data_ptr()), w.S_sel, w.n_sel, w.d, w.K, w.R, w.V, 1,
            vp(u.data_ptr()), None, vp(slot.data_ptr()), vp(score.data_ptr()),
            vp(flag.data_ptr()), vp(stream.cuda_stream))
    buf = torch.zeros(512 * 64, dtype=torch.int64)
    for _ in range(max(a.calls, 1)):
        torch.cuda.synchronize()
        if lib.dflash2_trace_read(vp(buf.data_ptr()), buf.numel() * 8, 1) != 0:
            raise RuntimeError("trace read failed")
        flush.zero_()
        if lib.dflash2_select(*args) != 0:
            raise RuntimeError(lib.dflash2_last_error().decode())
    torch.cuda.synchronize()
    if int(flag.item()) != 0:
        raise RuntimeError("device error flag set")
    if lib.dflash2_trace_read(vp(buf.data_ptr()), buf.numel() * 8, 0) != 0:
        raise RuntimeError("trace read failed")
    st = buf.view(512, 64)
    st = st[st[:, 0] > 0]
    t0 = int(st[:, 0].min())
    out = {"workload": w.name, "ctas": int(st.shape[0]), "us_after_first_entry": {}}
    for k, name in sorted(SLOTS.items()):
        col = st[:, k]
        col = col[col > 0]
        if col.numel():
            out["us_after_first_entry"][f"{k} {name}"] = round(float((col - t0).float().median()) / 1e3, 2)
    if a.json:
        print(json.dumps(out))
        return
    print(f"{w.name}: {out['ctas']} CTAs; median over CTAs, us after the first CTA's entry")
    for k, v in out["us_after_first_entry"].items():
        print(f"  {k:40s} {v:7.2f}")


if __name__ == "__main__":
    main()
