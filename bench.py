#!/usr/bin/env python
"""Benchmark of the CPR Gated DeltaNet hot path on one GB300 (or N independent GPUs).

One step = the whole hot path over the prefill workload (4 sequences x 4096 tokens,
16 query/key heads shared by 32 value heads, d = 128, C = 64, bf16 inputs):
    1. rollout prefill with a decode cache          (work list, boundary pass, chunks)
    2. 64 decode steps continuing those 4 sequences (one resynchronisation each),
       replayed from a CUDA graph
    3. trainer forward + backward on the same 16384 tokens
Tokens per step = 16384 (prefill) + 4 x 64 (decode) + 16384 (trainer).  `value` is
tokens/s over the whole step with inputs resident in HBM.  Per-stage times, a
256-slot decode measurement (the decode workload's shape: 256 x 32 heads of d = 128
states, 64 steps with one resync), per-kernel rooflines from CUDA events recorded by the
library on its launching stream, the end-to-end number through host buffers and the fp64
oracle timed on the host cores are reported in the same JSON line.

--impl reference times the fp64 CPU oracle (the only reference this operator has) on a
bounded sample of the same workload per step.

Multi-GPU: one process per GPU (torchrun).  Every rank runs its own copy of the workload
(independent sequences, no collective on the data path: weak scaling); rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "CPR GDN prefill & fwd+bwd tokens/s, decode µs/step; % HBM/TC roofline"
UNIT = "tokens/s"
WORKLOAD = "prefill"
DECODE_STEPS = 64
DECODE_SLOTS_BIG = 256
PEAK_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SMS, FP32_LANES, SM_MAX_MHZ = 152, 128, 2070.0

# DRAM bytes (read + write) per unit of work from one ncu capture of each kernel (summaries
# under profiles/), scaled to the benchmark's launch by the units it processes.  A figure is
# reported only while the kernel's source (its function text plus common.cuh) hashes to the
# value it had when the counters were taken; after any change it is null until recaptured.
NCU_TRAFFIC = {
    # 202,414,592 + 21,460,224 B for one 4096-token sequence x 32 value heads
    "k_intra": {"src_sha": "f0a18de335243fe2", "bytes_per_unit": (202414592 + 21460224) / (4096 * 32),
                "unit": "token-head"},
    # 541,331,968 + 482,812,160 B for the full 256-slot x 32-head launch (one-pass capture)
    "k_decode": {"src_sha": "e6c9318da9ca39cb", "bytes_per_unit": (541331968 + 482812160) / (256 * 32),
                 "unit": "slot-head"},
}
KERNEL_TEXT = {  # file, first line of the kernel, first line after it
    "k_intra": ("kernels_fwd.cu", "__global__ void __launch_bounds__(2 * D, 2) k_intra(",
                "static void launch_intra_t("),
    "k_decode": ("kernels_fwd.cu", "__global__ void __launch_bounds__(2 * D, 2) k_decode(",
                 "static void launch_decode_t("),
}


# ------------------------------------------------------------------ utilities ----
def src_sha(kernel: str) -> str:
    csrc = os.path.join(ROOT, "gated_deltanet_cpr_gb300", "csrc")
    f, first, after = KERNEL_TEXT[kernel]
    with open(os.path.join(csrc, f)) as fh:
        text = fh.read()
    i = text.index(first)
    body = text[i:text.index(after, i)]
    with open(os.path.join(csrc, "common.cuh")) as fh:
        common = fh.read()
    return hashlib.sha256((common + "\0" + body).encode()).hexdigest()[:16]


def ncu_traffic(kernel: str, units: int):
    rec = NCU_TRAFFIC[kernel]
    if rec["bytes_per_unit"] is None or rec["src_sha"] != src_sha(kernel):
        return None
    return rec["bytes_per_unit"] * units


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(PEAK_FALLBACK), "fallback"


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def shard_seed(rank: int) -> int:
    """Weak scaling: every rank draws its own independent copy of the workload."""
    return 1000 * rank


def reduce_max(value: float, world: int) -> float:
    """Max over ranks (the slowest rank defines the job's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock and throttle reasons; entering waits (up
    to 5 s) for the first sample so that the timed region is covered."""

    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = (bus_id or "").lower()
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"gdn_cpr_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        if self.proc is not None:
            t0 = time.time()
            while time.time() - t0 < 5.0 and self.proc.poll() is None:
                self.f.flush()
                if os.path.getsize(self.path) > 0:
                    break
                time.sleep(0.05)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()
        return False

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append(parts)
        if self.bus_id:
            mine = [r for r in rows if r[1].lower().endswith(self.bus_id[-12:])]
            rows = mine or rows
        if rows:
            idx0 = rows[0][0]
            rows = [r for r in rows if r[0] == idx0]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[2]) for r in rows if num(r[2]) is not None]
        mx = [num(r[3]) for r in rows if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max((num(r[4]) or 0.0) for r in rows)}


# ------------------------------------------------------------- CPU baseline ----
def oracle_rates(x, hv, fwd_tokens: int, bwd_tokens: int, threads: int):
    """Time the fp64 oracle (as it stands) on the first `fwd_tokens` / `bwd_tokens` tokens
    of the first sequence, all value heads.  Returns token-heads/s for forward and for
    backward (the backward recomputes its own forward)."""
    import oracle
    from gated_deltanet_cpr_gb300.synth import as_f64 as f

    def sl(n, L):
        return f(x[n][:L])

    t0 = time.perf_counter()
    oracle.fwd(sl("q", fwd_tokens), sl("k", fwd_tokens), sl("v", fwd_tokens), sl("g", fwd_tokens),
               sl("beta", fwd_tokens), [0, fwd_tokens], n_threads=threads)
    t_fwd = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.bwd(sl("q", bwd_tokens), sl("k", bwd_tokens), sl("v", bwd_tokens), sl("g", bwd_tokens),
               sl("beta", bwd_tokens), [0, bwd_tokens], sl("dout", bwd_tokens), n_threads=threads)
    t_bwd = time.perf_counter() - t0
    return fwd_tokens * hv / t_fwd, bwd_tokens * hv / t_bwd, t_fwd + t_bwd


def oracle_rates_all(x, hv, threads: int):
    """The oracle (as it stands) forward and backward over all sequences of x.  Returns
    token-heads/s for forward and for backward, and the wall time."""
    import oracle
    from gated_deltanet_cpr_gb300.synth import as_f64 as f

    cu = x["cu_seqlens"].numpy()
    T = int(cu[-1])
    t0 = time.perf_counter()
    oracle.fwd(f(x["q"]), f(x["k"]), f(x["v"]), f(x["g"]), f(x["beta"]), cu, n_threads=threads)
    t_fwd = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.bwd(f(x["q"]), f(x["k"]), f(x["v"]), f(x["g"]), f(x["beta"]), cu, f(x["dout"]),
               n_threads=threads)
    t_bwd = time.perf_counter() - t0
    return T * hv / t_fwd, T * hv / t_bwd, t_fwd + t_bwd


def step_tokens(w):
    T = w.total_tokens
    n_seq = len(w.lengths)
    return {"prefill": T, "decode": n_seq * DECODE_STEPS, "trainer": T}


def oracle_step_estimate(w, rate_fwd, rate_bwd):
    """Seconds the oracle would take for one whole step (linear in token-heads)."""
    tk = step_tokens(w)
    hv = w.h_v
    return ((tk["prefill"] + tk["decode"]) * hv / rate_fwd
            + tk["trainer"] * hv * (1.0 / rate_fwd + 1.0 / rate_bwd))


def threads_available():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- reference ----
def run_reference(args):
    """The fp64 CPU oracle as it stands, timed on the host cores.  Each step is a bounded
    sample of the benchmark step with the same mix of work (1/16 of every part): oracle
    forward over 1024 tokens (the prefill part), forward over the next 16 tokens (the decode
    part: the oracle's token recurrence is the decode step), forward and backward over 1024
    tokens (the trainer part), all 32 value heads of sequence 0.  value = the sample's tokens
    / its measured wall time; ms_per_step = that measured time (nothing is extrapolated)."""
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    import oracle
    from gated_deltanet_cpr_gb300 import synth
    from gated_deltanet_cpr_gb300.synth import as_f64 as f

    w = synth.workloads()[WORKLOAD]
    tk = step_tokens(w)
    frac = 16
    n_pre, n_dec, n_trn = tk["prefill"] // frac, tk["decode"] // frac, tk["trainer"] // frac
    x = synth.make_inputs([n_pre + n_dec], w.h_qk, w.h_v, w.d, dtype=w.dtype, seed=0, dout=True)
    a = {n: f(x[n]) for n in ("q", "k", "v", "g", "beta", "dout")}
    threads = threads_available()

    def sample_step():
        t0 = time.perf_counter()
        oracle.fwd(*(a[n][:n_pre] for n in ("q", "k", "v", "g", "beta")), [0, n_pre], n_threads=threads)
        oracle.fwd(*(a[n][n_pre:] for n in ("q", "k", "v", "g", "beta")), [0, n_dec], n_threads=threads)
        oracle.fwd(*(a[n][:n_trn] for n in ("q", "k", "v", "g", "beta")), [0, n_trn], n_threads=threads)
        oracle.bwd(*(a[n][:n_trn] for n in ("q", "k", "v", "g", "beta")), [0, n_trn], a["dout"][:n_trn],
                   n_threads=threads)
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        sample_step()
    times = [sample_step() for _ in range(args.steps)]
    sec = sum(times) / len(times)
    sample_tokens = n_pre + n_dec + n_trn
    value = sample_tokens / sec
    sample = (f"each step 1/{frac} of the benchmark step with its mix of work, all {w.h_v} value heads "
              f"of sequence 0: oracle fwd over {n_pre} tokens (prefill part), fwd over {n_dec} "
              f"tokens (decode part), fwd + bwd over {n_trn} tokens (trainer part); "
              f"{sample_tokens} tokens per step, measured wall time")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) inputs, q/k L2-normalised, beta=sigmoid, g=-softplus)",
            "config": step_config(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def step_config(w):
    tokens = step_tokens(w)
    return {"workload": w.name, "tokens_per_step": sum(tokens.values()), "stages": tokens,
            "l2": "inputs larger than L2 (step working set > 2 GB of HBM traffic)",
            "bwd_included": True}


# ---------------------------------------------------------------- CUDA arm ----
def run_cuda(args):
    import torch

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    dev = torch.device("cuda", local_rank if world > 1 else 0)
    torch.cuda.set_device(dev)

    from gated_deltanet_cpr_gb300 import api, synth

    api.load()
    P, peak_kind = peaks()
    w = synth.workloads()[WORKLOAD]
    C, d, hqk, hv = w.chunk, w.d, w.h_qk, w.h_v
    nseq = len(w.lengths)
    seed = shard_seed(rank)
    x = synth.make_inputs(w.lengths, hqk, hv, d, dtype=w.dtype, seed=seed, dout=True)
    # decode tokens (one per sequence per step)
    xd = synth.make_inputs([DECODE_STEPS * nseq], hqk, hv, d, dtype=w.dtype, seed=seed + 7)
    host = {n: x[n].pin_memory() for n in ("q", "k", "v", "g", "beta", "dout", "cu_seqlens")}
    t = {n: host[n].to(dev) for n in host}
    dq_in = {n: xd[n].view(DECODE_STEPS, nseq, *xd[n].shape[1:]).contiguous().to(dev)
             for n in ("q", "k", "v", "g", "beta")}
    cu_host = x["cu_seqlens"]
    T = w.total_tokens
    stream = torch.cuda.current_stream(dev)

    # resident buffers
    shp = api.make_shape(nseq, T, hqk, hv, d, C, torch.bfloat16, torch.bfloat16)
    ws_pre = api.alloc_workspace(api.workspace_bytes(shp, api.MODE_PREFILL, cu_host), dev)
    ws_fwd = api.alloc_workspace(api.workspace_bytes(shp, api.MODE_FWD, cu_host), dev)
    have_bwd = True
    try:
        ws_bwd = api.alloc_workspace(api.workspace_bytes(shp, api.MODE_BWD, cu_host), dev)
    except api.GdnError:
        have_bwd = False
        ws_bwd = None
    dshp = api.make_shape(nseq, nseq, hqk, hv, d, C, torch.bfloat16, torch.bfloat16)
    ws_dec = api.alloc_workspace(api.workspace_bytes(dshp, api.MODE_DECODE), dev)
    cache = api.Cache(nseq, hqk, hv, d, C, dtype=torch.bfloat16, device=dev)
    o_pre = torch.empty((T, hv, d), dtype=torch.bfloat16, device=dev)
    st_pre = torch.empty((nseq, hv, d, d), dtype=torch.float32, device=dev)
    o_fwd = torch.empty_like(o_pre)
    st_fwd = torch.empty_like(st_pre)
    n_chunks = sum((L + C - 1) // C for L in w.lengths)
    saved = torch.empty((n_chunks, hv, d, d), dtype=torch.float32, device=dev)
    o_dec = torch.empty((DECODE_STEPS, nseq, hv, d), dtype=torch.bfloat16, device=dev)
    slots = torch.arange(nseq, dtype=torch.int32, device=dev)
    grads = None

    def prefill_call(o=None):
        api.prefill(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], chunk=C,
                    cache=cache, cu_seqlens_host=cu_host, ws=ws_pre, o=o_pre if o is None else o,
                    state_out=st_pre)

    # every step's prefill leaves each sequence at position L, so decode step i of a step
    # starts at L + i: the host knows the positions (gdn_cpr_decode_step_pos)
    def decode_call(i, src=None):
        s_ = dq_in if src is None else src
        api.decode_step(s_["q"][i], s_["k"][i], s_["v"][i], s_["g"][i], s_["beta"][i], slots, cache,
                        ws=ws_dec, o=o_dec[i], pos_host=[L + i for L in w.lengths])

    def capture_decode(src):
        """A CUDA graph of the 64 decode steps reading their tokens from `src`."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(DECODE_STEPS):
                decode_call(i, src)
        return g

    def trainer_call(grad_out=None):
        nonlocal grads
        api.fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], chunk=C,
                cu_seqlens_host=cu_host, ws=ws_fwd, o=o_fwd, state_out=st_fwd, saved_bnd=saved)
        if have_bwd:
            grads = api.bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], saved,
                            t["dout"], chunk=C, cu_seqlens_host=cu_host, ws=ws_bwd,
                            want_dstate_in=True, out=grad_out)

    # the 64 decode steps as one CUDA graph (fixed pointers, device-side resync decision)
    prefill_call()
    for i in range(2):
        decode_call(i)
    torch.cuda.synchronize(dev)
    with api.Profiler(2) as cap_prof:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(DECODE_STEPS):
                decode_call(i)
    decode_kernels_per_replay = cap_prof.kernels

    tokens = step_tokens(w)
    step_tok = sum(tokens.values()) if have_bwd else tokens["prefill"] + tokens["decode"] + tokens["trainer"]

    def one_step(prof_pre, prof_fwd, ev):
        ev[0].record(stream)
        with prof_pre:
            prefill_call()
        ev[1].record(stream)
        graph.replay()
        ev[2].record(stream)
        with prof_fwd:
            trainer_call()
        ev[3].record(stream)

    mk = lambda: torch.cuda.Event(enable_timing=True)
    for _ in range(args.warmup):
        one_step(api.Profiler(6), api.Profiler(12), [mk() for _ in range(4)])
    torch.cuda.synchronize(dev)

    profs = [(api.Profiler(6), api.Profiler(12), [mk() for _ in range(4)]) for _ in range(args.steps)]
    start, end = mk(), mk()
    bus = getattr(torch.cuda.get_device_properties(dev), "pci_bus_id", None)
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(None if bus is None else str(bus)) as clk:
        start.record(stream)
        for pp, pf, ev in profs:
            one_step(pp, pf, ev)
        end.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    ms_local = start.elapsed_time(end) / args.steps
    ms = reduce_max(ms_local, world)
    value = world * step_tok / (ms * 1e-3)
    launches = sum(pp.kernels + pf.kernels for pp, pf, _ in profs) + args.steps * decode_kernels_per_replay

    stage_ms = {"prefill": statistics.mean(ev[0].elapsed_time(ev[1]) for _, _, ev in profs),
                "decode_64_steps": statistics.mean(ev[1].elapsed_time(ev[2]) for _, _, ev in profs),
                "trainer_fwd_bwd": statistics.mean(ev[2].elapsed_time(ev[3]) for _, _, ev in profs)}
    pre_k = [pp.stage_ms() for pp, _, _ in profs]
    names = ["worklist", "boundary_prepass", "boundary_chain", "intra_chunk", "cache_tail"]
    kern = {n: statistics.mean(s[i] for s in pre_k) for i, n in enumerate(names) if all(len(s) > i for s in pre_k)}
    bwd_k = [pf.stage_ms() for _, pf, _ in profs]
    bnames = ["bwd_worklist", "bwd_prep", "bwd_chain", "bwd_big_products", "bwd_gradients", "bwd_gqa_sum"]
    if have_bwd:
        kern.update({n: statistics.mean(s[i] for s in bwd_k) for i, n in enumerate(bnames)
                     if all(len(s) > i for s in bwd_k)})

    # dominant kernel: intra-chunk recurrence (FP32 ALU bound).  Algorithmic work in lane-ops:
    # 4 d^2 per token-head (the recurrence's decay multiply and three FMA per state element),
    # against one FP32 operation per lane per cycle on 152 SMs x 128 lanes at the maximum clock.
    intra_ms = kern["intra_chunk"]
    lane_ops = T * hv * 4 * d * d
    lane_peak = SMS * FP32_LANES * SM_MAX_MHZ * 1e6 / 1e12  # Tops/s
    ach_intra = lane_ops / (intra_ms * 1e-3) / 1e12
    flops_intra = T * hv * 6 * d * d  # the three FMA sweeps the scaled-state step executes
    fma_peak = 2 * lane_peak
    roofline = {"bound": "alu", "kernel": "k_intra (intra-chunk recurrence)", "achieved": ach_intra,
                "peak": lane_peak, "unit": "Tlane-op/s", "frac": ach_intra / lane_peak,
                "traffic": ncu_traffic("k_intra", T * hv),
                "peak_note": ("one FP32 lane-op per lane per cycle, 152 SMs x 128 lanes x 2070 MHz; "
                              "work 4 d^2 lane-ops per token-head (decay multiply + 3 FMA per state "
                              "element)"),
                "fma_flop": {"achieved": flops_intra / (intra_ms * 1e-3) / 1e12, "peak": fma_peak,
                             "unit": "TFLOP/s", "frac": flops_intra / (intra_ms * 1e-3) / 1e12 / fma_peak,
                             "note": ("the FMA FLOP the kernel executes: the decay is carried as a "
                                      "scalar scale of the state, so 3 FMA sweeps = 6 d^2 FLOP per "
                                      "token-head, against 2 FLOP per lane per cycle")}}
    chunk_heads_full = sum(L // C for L in w.lengths) * hv
    flops_bnd = chunk_heads_full * (6 * C * C * d + 4 * C * d * d)
    bnd_ms = kern["boundary_prepass"] + kern["boundary_chain"]
    tc_peak = float(P.get("bf16_tflops", PEAK_FALLBACK["bf16_tflops"]))
    hbm_peak = float(P.get("hbm_gbs", PEAK_FALLBACK["hbm_gbs"]))
    # algorithmic bytes of the boundary pass: K (per query/key head), V, g, beta read once,
    # the boundary state before every chunk written once (fp32 d x d)
    chunks = sum((L + C - 1) // C for L in w.lengths)
    bnd_bytes = (chunks * C * d * 2 * (hqk + hv) + chunks * hv * C * 4 * 2 + chunks * hv * d * d * 4)
    bnd_gbs = bnd_bytes / (bnd_ms * 1e-3) / 1e9
    boundary = {"bound": "hbm", "achieved": bnd_gbs, "peak": hbm_peak, "unit": "GB/s",
                "frac": bnd_gbs / hbm_peak, "algorithmic_bytes": bnd_bytes,
                "tensor": {"achieved": flops_bnd / (bnd_ms * 1e-3) / 1e12, "peak": tc_peak,
                           "unit": "TFLOP/s", "frac": flops_bnd / (bnd_ms * 1e-3) / 1e12 / tc_peak,
                           "flop": flops_bnd},
                "note": ("pre-pass + chain on tcgen05 (split-bf16 operands, fp32 accumulation in "
                         "TMEM); arithmetic intensity flop/algorithmic_bytes is below the bf16 "
                         "ridge point peak_TFLOP/s / peak_GB/s, so HBM bounds this pass")}

    # backward as a whole: inputs read once, gradients written once (algorithmic bytes)
    bwd_roof = None
    if have_bwd and grads is not None:
        bwd_ms = sum(kern.get(n, 0.0) for n in bnames)
        bwd_bytes = (sum(t[n].numel() * t[n].element_size() for n in ("q", "k", "v", "g", "beta", "dout"))
                     + saved.numel() * saved.element_size()
                     + sum(grads[n].numel() * grads[n].element_size()
                           for n in ("dq", "dk", "dv", "dg", "dbeta", "dstate_in")))
        bwd_gbs = bwd_bytes / (bwd_ms * 1e-3) / 1e9
        bwd_roof = {"bound": "hbm", "achieved": bwd_gbs, "peak": hbm_peak, "unit": "GB/s",
                    "frac": bwd_gbs / hbm_peak, "algorithmic_bytes": bwd_bytes, "ms": bwd_ms,
                    "note": "all backward kernels; the chunk-form workspace round trips are not "
                            "algorithmic bytes"}

    # the decode workload: 256 sequences prefilled with 2048 tokens, then 128 graph-replayed
    # decode steps, per kernel and per step
    dec = bench_decode_big(api, synth, torch, dev, w, P, seed)
    # the trainer workload (8 packed varlen sequences) and the long-context prefill
    trainer_cfg = bench_trainer_workload(api, synth, torch, dev, seed)
    longctx_cfg = bench_longctx_workload(api, synth, torch, dev, seed)

    # prefill continued from a cache: chunked prefill and multi-token decode
    cont = bench_continue(api, synth, torch, dev, w, seed, stage_ms["prefill"])

    # end to end through host buffers: H2D inputs each step, D2H results each step
    e2e = bench_e2e(api, torch, dev, w, host, xd, args, prefill_call, graph, capture_decode, trainer_call,
                    t, dq_in, o_pre, o_dec, lambda: grads, step_tok, world, ms)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) inputs, q/k L2-normalised, beta=sigmoid, g=-softplus)",
            "config": dict(step_config(w), bwd_included=have_bwd),
            "stage_ms": stage_ms, "kernel_ms": kern, "roofline": roofline,
            "boundary_roofline": boundary, "bwd_roofline": bwd_roof, "decode": dec,
            "continue": cont, "trainer_workload": trainer_cfg, "longctx_workload": longctx_cfg,
            "e2e": e2e,
            "gpu_launches": launches, "clocks": clk.summary(),
            "peaks_source": f"{peak_kind} (MEASURED_PEAKS.json)" if peak_kind == "measured" else peak_kind}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = threads_available()
        rf, rb, dt = oracle_rates_all(x, hv, threads)
        est = oracle_step_estimate(w, rf, rb)
        rf1, rb1, dt1 = oracle_rates(x, hv, 512, 256, 1)
        est1 = oracle_step_estimate(w, rf1, rb1)
        line["cpu_baseline"] = {
            "value": step_tok / est, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": (f"oracle fwd and oracle bwd over the whole prefill workload "
                       f"({T} tokens x {hv} heads each, {dt:.1f} s wall on {threads} threads); "
                       f"step time = those rates applied to the step's token-heads"),
            "single_core": {"value": step_tok / est1, "unit": UNIT, "cores": 1,
                            "sample": (f"oracle fwd over 512 tokens and bwd over 256 tokens x {hv} "
                                       f"heads of sequence 0 on one thread ({dt1:.1f} s wall); step "
                                       f"time = those rates applied to the step's token-heads")}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def bench_decode_big(api, synth, torch, dev, w, P, seed):
    """The decode workload: 256 sequences, each first prefilled with 2048 tokens (through
    gdn_cpr_prefill with a cache, 64 sequences per call), then 128 decode steps of one token
    per sequence with a resynchronisation every 64 tokens (the steps whose token is the
    sequence's 2112th and 2176th), replayed from one CUDA graph.  Inputs are drawn on the
    device from seeded generators (the same distributions as the other workloads)."""
    wd = synth.workloads()["decode"]
    N, L0, M = len(wd.lengths), wd.lengths[0], wd.decode_steps
    C, d, hqk, hv = wd.chunk, wd.d, wd.h_qk, wd.h_v
    cache = api.Cache(N, hqk, hv, d, C, dtype=torch.bfloat16, device=dev)
    B = 64
    for b0 in range(0, N, B):
        xp = synth.make_inputs([L0] * B, hqk, hv, d, dtype=wd.dtype, seed=seed + 31 + b0, device=dev)
        sl = torch.arange(b0, b0 + B, dtype=torch.int32, device=dev)
        api.prefill(xp["q"], xp["k"], xp["v"], xp["g"], xp["beta"], xp["cu_seqlens"].to(dev), chunk=C,
                    cache=cache, slot_of_seq=sl, cu_seqlens_host=xp["cu_seqlens"], want_state=False)
        torch.cuda.synchronize(dev)
        del xp
    xd = synth.make_inputs([M * N], hqk, hv, d, dtype=wd.dtype, seed=seed + 13, device=dev)
    din = {n: xd[n].view(M, N, *xd[n].shape[1:]) for n in ("q", "k", "v", "g", "beta")}
    slots = torch.arange(N, dtype=torch.int32, device=dev)
    shp = api.make_shape(N, N, hqk, hv, d, C, torch.bfloat16, torch.bfloat16)
    ws = api.alloc_workspace(api.workspace_bytes(shp, api.MODE_DECODE), dev)
    o = torch.empty((M, N, hv, d), dtype=torch.bfloat16, device=dev)
    saved = {n: getattr(cache, n).clone() for n in api.Cache.TENSORS}

    def call(i):
        api.decode_step(din["q"][i], din["k"][i], din["v"][i], din["g"][i], din["beta"][i],
                        slots, cache, ws=ws, o=o[i], pos_host=[L0 + i] * N)

    def reset():
        for n in api.Cache.TENSORS:
            getattr(cache, n).copy_(saved[n])

    # per-kernel times from the library's stage events (direct launches)
    reset()
    per = []
    for i in range(M):
        prof = api.Profiler(5)
        with prof:
            call(i)
        per.append(prof)
    torch.cuda.synchronize(dev)
    stages = [p.stage_ms() for p in per]
    resync_steps = [i for i in range(M) if (L0 + i + 1) % C == 0]
    normal = [s for i, s in enumerate(stages) if i not in resync_steps]
    step_k3 = statistics.median(s[0] for s in normal)
    step_p50 = statistics.median(sum(s) for s in normal)
    resync_ms = [sum(stages[i]) for i in resync_steps]
    # graph replay of all 128 steps
    reset()
    call(0)
    reset()
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(M):
            call(i)
    times = []
    for _ in range(3):
        reset()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1))
    us_per_step = statistics.median(times) * 1e3 / M
    # K3 algorithmic bytes: state read+write, q,k per qk head, v, o, tail appends, g, beta
    bpe = 2
    bytes_k3 = (N * hv * d * d * 4 * 2 + N * hqk * d * bpe * 2 + N * hv * d * bpe
                + N * hv * d * bpe + N * hqk * d * bpe + N * hv * d * bpe + N * hv * 4 * 4)
    hbm = float(P.get("hbm_gbs", PEAK_FALLBACK["hbm_gbs"]))
    ach = bytes_k3 / (step_k3 * 1e-3) / 1e9
    return {"workload": wd.name, "slots": N, "heads": hv, "d": d, "steps": M,
            "start_state": f"a {L0}-token prefill of every sequence into the cache",
            "us_per_step_mean": us_per_step, "us_per_step_p50": step_p50 * 1e3,
            "us_token_step_kernel_median": step_k3 * 1e3,
            "resync_steps": len(resync_steps),
            "us_resync_step": statistics.mean(resync_ms) * 1e3,
            "us_resync_stages": dict(zip(("token_step", "resync", "advance"),
                                         (x * 1e3 for x in stages[resync_steps[0]]))),
            "tokens_per_s": N / (us_per_step * 1e-6),
            "roofline": {"bound": "hbm", "kernel": "k_decode (token step)", "achieved": ach,
                         "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                         "traffic": ncu_traffic("k_decode", N * hv),
                         "algorithmic_bytes_per_launch": bytes_k3}}


def bench_trainer_workload(api, synth, torch, dev, seed):
    """Trainer forward + backward on the trainer workload (8 packed sequences, lengths
    uniform in [512, 8192]), all six gradients including state_in's.  Inputs drawn on the
    device from seeded generators."""
    wt = synth.workloads()["trainer"]
    C, d, hqk, hv = wt.chunk, wt.d, wt.h_qk, wt.h_v
    x = synth.make_inputs(wt.lengths, hqk, hv, d, dtype=wt.dtype, seed=seed + 41, dout=True, device=dev)
    cu_host = x["cu_seqlens"]
    cu = cu_host.to(dev)
    N, T = len(wt.lengths), wt.total_tokens
    shp = api.make_shape(N, T, hqk, hv, d, C, torch.bfloat16, torch.bfloat16)
    ws_f = api.alloc_workspace(api.workspace_bytes(shp, api.MODE_FWD, cu_host), dev)
    ws_b = api.alloc_workspace(api.workspace_bytes(shp, api.MODE_BWD, cu_host), dev)
    nch = sum((L + C - 1) // C for L in wt.lengths)
    saved = torch.empty((nch, hv, d, d), dtype=torch.float32, device=dev)
    o = torch.empty((T, hv, d), dtype=torch.bfloat16, device=dev)
    st = torch.empty((N, hv, d, d), dtype=torch.float32, device=dev)
    mk = lambda: torch.cuda.Event(enable_timing=True)
    res = []
    for rep in range(6):
        e = [mk(), mk(), mk()]
        e[0].record()
        api.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, chunk=C, cu_seqlens_host=cu_host,
                ws=ws_f, o=o, state_out=st, saved_bnd=saved)
        e[1].record()
        api.bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, saved, x["dout"], chunk=C,
                cu_seqlens_host=cu_host, ws=ws_b, want_dstate_in=True)
        e[2].record()
        torch.cuda.synchronize(dev)
        if rep >= 2:
            res.append((e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2])))
    f_ms = statistics.median(r[0] for r in res)
    b_ms = statistics.median(r[1] for r in res)
    return {"workload": wt.name, "lengths": wt.lengths, "tokens": T, "fwd_ms": f_ms, "bwd_ms": b_ms,
            "ms": f_ms + b_ms, "tokens_per_s": T / ((f_ms + b_ms) * 1e-3)}


def bench_longctx_workload(api, synth, torch, dev, seed):
    """Rollout prefill of the long-context workload: 64 sequences with lengths log-uniform in
    [128, 32768] in one call.  Inputs drawn on the device from seeded generators."""
    wl = synth.workloads()["longctx"]
    C, d, hqk, hv = wl.chunk, wl.d, wl.h_qk, wl.h_v
    x = synth.make_inputs(wl.lengths, hqk, hv, d, dtype=wl.dtype, seed=seed + 51, device=dev)
    cu_host = x["cu_seqlens"]
    cu = cu_host.to(dev)
    N, T = len(wl.lengths), wl.total_tokens
    shp = api.make_shape(N, T, hqk, hv, d, C, torch.bfloat16, torch.bfloat16)
    ws = api.alloc_workspace(api.workspace_bytes(shp, api.MODE_PREFILL, cu_host), dev)
    o = torch.empty((T, hv, d), dtype=torch.bfloat16, device=dev)
    st = torch.empty((N, hv, d, d), dtype=torch.float32, device=dev)
    times = []
    for rep in range(4):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        api.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, chunk=C, cu_seqlens_host=cu_host,
                    ws=ws, o=o, state_out=st)
        e1.record()
        torch.cuda.synchronize(dev)
        if rep >= 1:
            times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    return {"workload": wl.name, "sequences": N, "tokens": T, "longest": max(wl.lengths), "ms": ms,
            "tokens_per_s": T / (ms * 1e-3)}


def bench_continue(api, synth, torch, dev, w, seed, prefill_ms):
    """Prefill continued from a cache: (1) the prefill workload's sequences fed in unaligned
    pieces after a first prefill (1000 + 1100 + 1000 + 996 tokens), the continued pieces timed;
    (2) 256 slots extended by 4 tokens per call (multi-token decode).  Both bit-identical to
    one prefill (tests/test_gpu_continue.py).  The cache is restored between repetitions,
    outside the timed region."""
    C, d, hqk, hv = w.chunk, w.d, w.h_qk, w.h_v
    nseq, L = len(w.lengths), w.lengths[0]
    cuts = [0, 1000, 2100, 3100, L]
    x = synth.make_inputs(w.lengths, hqk, hv, d, dtype=w.dtype, seed=seed + 21)
    cu = x["cu_seqlens"].tolist()
    names = ("q", "k", "v", "g", "beta")

    def piece(a, b):
        t = {n: torch.cat([x[n][cu[i] + a:cu[i] + b] for i in range(nseq)]).to(dev) for n in names}
        return t, synth.cu_seqlens_of([b - a] * nseq)

    cache = api.Cache(nseq, hqk, hv, d, C, dtype=torch.bfloat16, device=dev)
    slots = torch.arange(nseq, dtype=torch.int32, device=dev)
    t0, cu0 = piece(0, cuts[1])
    api.prefill(t0["q"], t0["k"], t0["v"], t0["g"], t0["beta"], cu0.to(dev), chunk=C, cache=cache,
                slot_of_seq=slots, cu_seqlens_host=cu0)
    start_state = {n: getattr(cache, n).clone() for n in api.Cache.TENSORS}
    pieces = [piece(cuts[i], cuts[i + 1]) for i in range(1, len(cuts) - 1)]
    plans = []
    for (tp, cup), a in zip(pieces, cuts[1:-1]):
        shp = api.make_shape(nseq, int(cup[-1]), hqk, hv, d, C, torch.bfloat16, torch.bfloat16)
        plans.append((tp, cup, cup.to(dev), [a] * nseq,
                      api.alloc_workspace(api.workspace_bytes(shp, api.MODE_CONTINUE, cup), dev),
                      torch.empty((int(cup[-1]), hv, d), dtype=torch.bfloat16, device=dev)))
    times = []
    for rep in range(4):
        for n in api.Cache.TENSORS:
            getattr(cache, n).copy_(start_state[n])
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for tp, cup, cud, pos, ws, o in plans:
            api.prefill_continue(tp["q"], tp["k"], tp["v"], tp["g"], tp["beta"], cud, slots, cache,
                                 pos_host=pos, cu_seqlens_host=cup, ws=ws, o=o)
        e1.record()
        torch.cuda.synchronize(dev)
        if rep > 0:
            times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    tok = nseq * (L - cuts[1])
    # multi-token decode: 256 slots, 4 tokens each per call
    N, K = DECODE_SLOTS_BIG, 4
    dc = api.Cache(N, hqk, hv, d, C, dtype=torch.bfloat16, device=dev)
    gen = torch.Generator(device=dev).manual_seed(seed + 23)
    dc.s_run.normal_(generator=gen).mul_(0.05)
    dc.s_bnd.copy_(dc.s_run)
    dc.tail_k.normal_(generator=gen).mul_(0.09)
    dc.tail_v.normal_(generator=gen)
    dc.tail_g.uniform_(-1.5, -0.1, generator=gen)
    dc.tail_beta.uniform_(0.2, 0.8, generator=gen)
    dc.pos.fill_(2048 + 30)
    xd = synth.make_inputs([K] * N, hqk, hv, d, dtype=w.dtype, seed=seed + 25)
    td = {n: xd[n].to(dev) for n in names}
    cud = xd["cu_seqlens"]
    dslots = torch.arange(N, dtype=torch.int32, device=dev)
    shp = api.make_shape(N, N * K, hqk, hv, d, C, torch.bfloat16, torch.bfloat16)
    wsd = api.alloc_workspace(api.workspace_bytes(shp, api.MODE_CONTINUE, cud), dev)
    od = torch.empty((N * K, hv, d), dtype=torch.bfloat16, device=dev)
    saved = {n: getattr(dc, n).clone() for n in api.Cache.TENSORS}
    dt = []
    for rep in range(6):
        for n in api.Cache.TENSORS:
            getattr(dc, n).copy_(saved[n])
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        api.prefill_continue(td["q"], td["k"], td["v"], td["g"], td["beta"], cud.to(dev), dslots, dc,
                             pos_host=[2048 + 30] * N, cu_seqlens_host=cud, ws=wsd, o=od)
        e1.record()
        torch.cuda.synchronize(dev)
        if rep > 0:
            dt.append(e0.elapsed_time(e1))
    us = statistics.median(dt) * 1e3
    return {"chunked_prefill": {"pieces": [b - a for a, b in zip(cuts[1:-1], cuts[2:])], "sequences": nseq,
                                "tokens": tok, "ms": ms, "tokens_per_s": tok / (ms * 1e-3),
                                "one_shot_prefill_tokens_per_s": nseq * L / (prefill_ms * 1e-3)},
            "multi_token_decode": {"slots": N, "tokens_per_slot": K, "pos_mod_C": 30,
                                   "us_per_call": us, "tokens_per_s": N * K / (us * 1e-6)}}


def bench_e2e(api, torch, dev, w, host, xd, args, prefill_call, graph, capture_decode, trainer_call, t, dq_in,
              o_pre, o_dec, get_grads, step_tok, world, compute_ms):
    """Same step through the public API with host buffers: every step copies its inputs from
    pinned host memory and reads its results back, pipelined as a serving or training loop
    would run it: step i + 1's inputs (prefill / trainer tokens and the decode tokens) go up on
    a copy stream (into the second of two input buffers, the decode steps replayed from one
    CUDA graph per buffer) while step i computes, and every result comes back on the same copy
    stream (or, with --e2e-copy-streams 2, on a second one) as soon as its kernels finish: one
    stream keeps the two directions from contending for the host link (measured: the copies
    of a step take the isolated copy rates' time on one stream, about 15% more on two on a
    quiet box and 1.7 times as much on a busy one); the prefill output and the gradients alternate
    between two sets of buffers, so a step's compute never waits for the previous step's
    read-back of them; the timed region opens before the first input copy and closes after
    the last read-back."""
    nseq = len(w.lengths)
    dhost = {n: xd[n].view(DECODE_STEPS, nseq, *xd[n].shape[1:]).contiguous().pin_memory()
             for n in ("q", "k", "v", "g", "beta")}
    h2d = sum(v.numel() * v.element_size() for v in host.values()) + \
        sum(v.numel() * v.element_size() for v in dhost.values())

    o_pre_bufs = [o_pre, torch.empty_like(o_pre)]
    cur = {"pre": o_pre, "trn": None}

    def result_tensors(part):
        if part == "pre":
            return {"o_prefill": cur["pre"]}
        if part == "dec":
            return {"o_decode": o_dec}
        gr = get_grads() if cur["trn"] is None else cur["trn"]
        return {} if gr is None else {n: gr[n] for n in ("dq", "dk", "dv", "dg", "dbeta", "dstate_in")}

    comp = torch.cuda.current_stream(dev)
    up = torch.cuda.Stream(dev)
    down = up if args.e2e_copy_streams == 1 else torch.cuda.Stream(dev)
    t0 = dict(t)
    bufs = [t0, {n: torch.empty_like(v) for n, v in t0.items()}]
    dq_bufs = [dq_in, {n: torch.empty_like(v) for n, v in dq_in.items()}]
    graphs = [graph, capture_decode(dq_bufs[1])]
    trainer_call()  # so that the gradient tensors exist for sizing the host buffers
    torch.cuda.synchronize(dev)
    grad_bufs = [{n: torch.empty_like(v) for n, v in get_grads().items()} for _ in range(2)]
    res_host = {n: torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                for part in ("pre", "dec", "trn") for n, v in result_tensors(part).items()}
    d2h = sum(v.numel() * v.element_size() for v in res_host.values())
    mk = torch.cuda.Event
    up_done, in_free, pre_free, trn_free = [mk(), mk()], [mk(), mk()], [mk(), mk()], [mk(), mk()]
    produced = {p: mk() for p in ("pre", "dec", "trn")}
    read_back = {p: mk() for p in ("pre", "dec", "trn")}

    copy_ev = {"up": [], "down": []}  # (start, end) of every upload / read-back of the timed run

    def timed(kind, stream):
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        copy_ev[kind].append((a_, b_))
        return a_, b_

    def upload(b, after=None):
        with torch.cuda.stream(up):
            if after is not None:
                up.wait_event(after)
            up.wait_event(in_free[b])
            ea, eb = timed("up", up)
            ea.record(up)
            for n in host:
                bufs[b][n].copy_(host[n], non_blocking=True)
            for n in dhost:
                dq_bufs[b][n].copy_(dhost[n], non_blocking=True)
            eb.record(up)
            up_done[b].record(up)

    def download(part):
        with torch.cuda.stream(down):
            down.wait_event(produced[part])
            ea, eb = timed("down", down)
            ea.record(down)
            for n, v in result_tensors(part).items():
                v.record_stream(down)
                res_host[n].copy_(v, non_blocking=True)
            eb.record(down)
            read_back[part].record(down)

    def run(n_steps, e_start=None):
        upload(0, e_start)
        for i in range(n_steps):
            b = i % 2
            comp.wait_event(up_done[b])
            if i + 1 < n_steps:
                upload(1 - b)
            t.update(bufs[b])
            cur["pre"] = o_pre_bufs[b]
            comp.wait_event(pre_free[b])  # the read-back of this buffer two steps ago
            prefill_call(cur["pre"])
            produced["pre"].record(comp)
            download("pre")
            pre_free[b].record(down)
            comp.wait_event(read_back["dec"])
            graphs[b].replay()
            produced["dec"].record(comp)
            download("dec")
            cur["trn"] = grad_bufs[b]
            comp.wait_event(trn_free[b])  # the read-back of this set two steps ago
            trainer_call(cur["trn"])
            produced["trn"].record(comp)
            in_free[b].record(comp)
            download("trn")
            trn_free[b].record(down)
        comp.wait_stream(down)

    run(max(1, args.warmup))
    torch.cuda.synchronize(dev)
    barrier(world)
    copy_ev["up"].clear()
    copy_ev["down"].clear()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    run(args.steps, e0)
    e1.record(comp)
    torch.cuda.synchronize(dev)
    barrier(world)
    # how long the copies of a step took while the step computed (against the serial rates
    # measured below, this shows whether the box slowed them down)
    up_ms = sum(a_.elapsed_time(b_) for a_, b_ in copy_ev["up"]) / args.steps
    down_ms = sum(a_.elapsed_time(b_) for a_, b_ in copy_ev["down"]) / args.steps
    t.update(t0)
    # every step recomputes the same results (bit-exact), so the host copies must equal the
    # device results: a race between the streams would show here
    for part in ("pre", "dec", "trn"):
        for n, v in result_tensors(part).items():
            if not torch.equal(res_host[n], v.cpu()):
                raise RuntimeError(f"pipelined end-to-end read-back of {n} differs from the device result")
    ms = reduce_max(e0.elapsed_time(e1) / args.steps, world)
    # the machine's host<->device copy rates (pinned host memory, one 256 MiB copy each way,
    # best of 3) and what the step's copies cost at those rates if nothing overlapped
    hb = torch.empty(1 << 28, dtype=torch.uint8, pin_memory=True)
    db = torch.empty(1 << 28, dtype=torch.uint8, device=dev)
    bw = {}
    for name, dst, src in (("h2d", db, hb), ("d2h", hb, db)):
        best = None
        for _ in range(3):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(comp)
            dst.copy_(src, non_blocking=True)
            c1.record(comp)
            torch.cuda.synchronize(dev)
            best = c0.elapsed_time(c1) if best is None else min(best, c0.elapsed_time(c1))
        bw[name] = hb.numel() / (best * 1e-3) / 1e9
    del hb, db
    copy_ms = (h2d / bw["h2d"] + d2h / bw["d2h"]) / 1e6
    return {"value": world * step_tok / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "h2d_gbs": bw["h2d"], "d2h_gbs": bw["d2h"], "copy_ms_per_step_serial": copy_ms,
            "h2d_ms_per_step_during_run": up_ms, "d2h_ms_per_step_during_run": down_ms,
            "exposed_ms_per_step": ms - compute_ms,
            "copy_streams": args.e2e_copy_streams,
            "pipelined": "inputs of step i+1 uploaded during step i (two input buffers); "
                         + ("results read back on a second copy stream as each part finishes"
                            if args.e2e_copy_streams == 2 else
                            "results read back on the same copy stream, after it, as each part finishes")}


def run_ncu_case(args):
    """Small, fixed cases for ncu captures (a few hundred MB on the device):
    prefill   one 4096-token sequence, 16/32 heads, d=128, C=64, bf16: three prefills
    decode    64 slots x 32 heads of 128x128 states: three decode steps (no resync)
    decode256 the decode workload's 256 slots x 32 heads: three decode steps (no resync), for
              one-pass DRAM counters of the full-size launch
    resync64  64 slots x 32 heads whose every step completes a chunk: three decode steps, each
              with its resync (k_resync_fused_tc)
    bwd       one 4096-token sequence: two trainer forward + backward passes
    """
    import torch

    from gated_deltanet_cpr_gb300 import api, synth

    dev = torch.device("cuda", 0)
    w = synth.workloads()[WORKLOAD]
    if args.ncu_case == "bwd":
        x = synth.make_inputs([4096], w.h_qk, w.h_v, w.d, dtype=w.dtype, seed=0, dout=True)
        t = {n: x[n].to(dev) for n in ("q", "k", "v", "g", "beta", "cu_seqlens", "dout")}
        for _ in range(2):
            _, _, saved = api.fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"],
                                  chunk=w.chunk, cu_seqlens_host=x["cu_seqlens"])
            api.bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], saved, t["dout"],
                    chunk=w.chunk, cu_seqlens_host=x["cu_seqlens"])
    elif args.ncu_case == "prefill":
        x = synth.make_inputs([4096], w.h_qk, w.h_v, w.d, dtype=w.dtype, seed=0)
        t = {n: x[n].to(dev) for n in ("q", "k", "v", "g", "beta", "cu_seqlens")}
        for _ in range(3):
            api.prefill(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], chunk=w.chunk,
                        cu_seqlens_host=x["cu_seqlens"])
    else:
        N = 256 if args.ncu_case == "decode256" else 64
        p0 = 2047 if args.ncu_case == "resync64" else 2048
        cache = api.Cache(N, w.h_qk, w.h_v, w.d, w.chunk, dtype=torch.bfloat16, device=dev)
        cache.s_run.normal_()
        cache.s_bnd.normal_().mul_(0.05)
        cache.tail_k.normal_().mul_(0.09)
        cache.tail_v.normal_()
        cache.tail_g.uniform_(-1.5, -0.1)
        cache.tail_beta.uniform_(0.2, 0.8)
        cache.pos.fill_(p0)
        x = synth.make_inputs([N], w.h_qk, w.h_v, w.d, dtype=w.dtype, seed=0)
        t = {n: x[n].to(dev) for n in ("q", "k", "v", "g", "beta")}
        slots = torch.arange(N, dtype=torch.int32, device=dev)
        for _ in range(3):
            cache.pos.fill_(p0)
            api.decode_step(t["q"], t["k"], t["v"], t["g"], t["beta"], slots, cache)
    torch.cuda.synchronize(dev)
    print(json.dumps({"ncu_case": args.ncu_case, "ok": True}))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-copy-streams", type=int, choices=[1, 2], default=1,
                    help="end-to-end run: uploads and read-backs on one copy stream (default) or "
                         "on two (concurrent directions, which contend for the host link)")
    ap.add_argument("--ncu-case", choices=["prefill", "decode", "decode256", "resync64", "bwd"], default=None,
                    help="run a small fixed case for an ncu capture and exit")
    args = ap.parse_args(argv)
    if args.ncu_case:
        return run_ncu_case(args)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_cuda(args)


if __name__ == "__main__":
    sys.exit(main())
