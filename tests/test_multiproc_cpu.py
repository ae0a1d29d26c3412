"""Host-side logic of the N > 1 benchmark path on CPU with gloo, world size 2:
each rank gets its own sequences, the timing reduction is a max over ranks,
and the reference arm runs on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    from dflash2_draft_head_gb300 import synth
    from dflash2_draft_head_gb300.workloads import Workload
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w0 = Workload(name="t", S=2, n=8, C=64, T=4, G=4, d=64, R=16, V=100, K=4, dtype="bf16",
                  S_sel=2, n_sel=8, seed=5)
    w = bench.rank_workload(w0, rank)
    x = synth.conv_inputs(w)["x"]
    sums = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(sums, torch.tensor([float(x.double().sum())], dtype=torch.float64))
    m = bench.max_over_ranks(1.5 + rank, world)
    q.put((rank, [float(s) for s in sums], m, w.seed))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_sharding_and_max_timing():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, sums0, m0, seed0), (r1, sums1, m1, seed1) = res
    assert sums0 == sums1 and sums0[0] != sums0[1]      # distinct sequences per rank
    assert m0 == m1 == 2.5                               # max over ranks
    assert seed0 != seed1


def test_reference_arm_nonzero_rank_exits_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                       env=env, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_rank0_prints_contract_line():
    """Rank 0 of the reference arm times the oracle and prints one JSON line
    with the keys the benchmark contract asks for."""
    import json
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_fp32", "--steps", "2", "--warmup", "1",
                        "--ref-seconds", "1"], capture_output=True, text=True,
                       env=env, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny_fp32"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
