"""The N > 1 path of bench.py on CPU with gloo (world size 2): per-rank step
times reduce to the max over ranks, and a torchrun launch prints exactly one
JSON line from rank 0 (the reference arm, which needs no GPU)."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    got = bench.max_over_ranks([1.5 + rank, 10.0 - rank], dist)
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0] == res[1] == [2.5, 10.0]


def test_torchrun_two_ranks_one_json_line():
    env = dict(os.environ, WNA16_BENCH_BACKEND="gloo", OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1", "--workload", "tiny_w2",
           "--oracle-seconds", "0.05"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"


def _ep_worker(rank, world, port, q):
    """Rank `rank` holds experts [rank*E/2, (rank+1)*E/2): the oracle's partial
    for them, summed across the two ranks with gloo and rounded to BF16."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import oracle
    import synth
    w = synth.get("tiny_w2")
    inp = synth.make_all(w, 0)
    _, _, y = oracle.forward(inp["x"], inp["ids"], inp["weights"], inp["w13_packed"], inp["w13_scales"],
                             inp["w2_packed"], inp["w2_scales"], bits=w.bits, group_size=w.g13,
                             group_size_w2=w.g2, swiglu_limit=w.swiglu_limit, return_intermediates=True)
    half = w.E // world
    part = torch.from_numpy(oracle.combine_partial(inp["ids"], inp["weights"], y, (rank * half, (rank + 1) * half)))
    dist.all_reduce(part, op=dist.ReduceOp.SUM)
    out = part.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    q.put((rank, out.tobytes()))
    dist.destroy_process_group()


def test_expert_parallel_sum_gloo():
    """Two gloo ranks each run the oracle's expert-parallel partial for half the
    experts; the all-reduced sum, rounded to BF16, is the oracle's
    expert-parallel profile (partials summed in rank order) bit for bit -- with
    two ranks the fp32 sum has one addition, so its order cannot differ."""
    import numpy as np
    import oracle
    import synth
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_ep_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    w = synth.get("tiny_w2")
    inp = synth.make_all(w, 0)
    _, _, y = oracle.forward(inp["x"], inp["ids"], inp["weights"], inp["w13_packed"], inp["w13_scales"],
                             inp["w2_packed"], inp["w2_scales"], bits=w.bits, group_size=w.g13,
                             group_size_w2=w.g2, swiglu_limit=w.swiglu_limit, return_intermediates=True)
    parts = [oracle.combine_partial(inp["ids"], inp["weights"], y, (0, w.E // 2)),
             oracle.combine_partial(inp["ids"], inp["weights"], y, (w.E // 2, w.E))]
    profile = oracle.sum_partials(parts)
    for r in (0, 1):
        got = np.frombuffer(res[r], np.uint16).reshape(profile.shape)
        assert np.array_equal(got, profile)
