"""The multi-GPU path's host logic on CPU: two ranks over gloo (world size 2).

The path shards by independent sequences (weak scaling) and has no collective on the data;
what crosses ranks is only the benchmark's own bookkeeping, which is tested here:
- every rank reads its rank / local rank / world size from the launcher's environment and
  draws its own, distinct copy of the workload;
- the step time is the maximum over ranks, the same on every rank, and the barrier lets no
  rank past until all have reached it;
- the whole-job value counts the tokens of all ranks;
- under torchrun the oracle reference arm runs on rank 0 alone, which prints exactly one
  JSON line, and the other rank exits 0 without work.
"""
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, lr, w = bench.dist_env()
    seed = bench.shard_seed(r)
    # a rank-dependent "step time": the job's time is the slowest rank's
    ms_local = 10.0 + 7.5 * r
    ms = bench.reduce_max(ms_local, w)
    # rank 1 arrives late at the barrier; rank 0 must not pass before it
    if r == 1:
        time.sleep(0.5)
    t_before = time.time()
    bench.barrier(w)
    t_after = time.time()
    from gated_deltanet_cpr_gb300 import synth

    wl = synth.workloads()["prefill"]
    x = synth.make_inputs(wl.lengths[:1], wl.h_qk, wl.h_v, wl.d, dtype=wl.dtype, seed=seed)
    step_tok = sum(bench.step_tokens(wl).values())
    value = w * step_tok / (ms * 1e-3)
    q.put({"rank": r, "local_rank": lr, "world": w, "seed": seed, "ms": ms, "value": value,
           "waited": t_after - t_before, "q0": float(x["q"].float()[0, 0, 0])})
    dist.destroy_process_group()


def test_two_gloo_ranks_bookkeeping():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in range(2):
        d = q.get(timeout=240)
        res[d["rank"]] = d
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(res) == [0, 1]
    assert all(res[r]["world"] == 2 and res[r]["local_rank"] == r for r in (0, 1))
    # independent shards: distinct seeds and distinct inputs
    assert res[0]["seed"] != res[1]["seed"]
    assert res[0]["q0"] != res[1]["q0"]
    # max over ranks, identical everywhere
    assert res[0]["ms"] == res[1]["ms"] == 17.5
    assert res[0]["value"] == res[1]["value"]
    # rank 0 waited at the barrier for the late rank 1
    assert res[0]["waited"] >= 0.3


def test_reference_arm_rank0_only():
    port = free_port()
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
