"""GPU parity of the trainer backward (gdn_cpr_bwd) against the fp64 oracle's hand-derived
reverse recurrence (itself pinned by central finite differences in test_oracle_pins.py).

Gradient of loss = <dO, o> + <dstate_out, state_out> with respect to q, k, v, g, beta and
state_in.  Tolerance per tensor: max|GPU - oracle| / max|oracle|, <= 2e-3 for bf16 inputs
and <= 1e-5 for fp32 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_cpr_gb300 import synth
from helpers import f64, rel_err, to_dev

pytestmark = pytest.mark.gpu

TOL = {synth.F32: 1e-5, synth.BF16: 2e-3}
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dstate_in")


def gpu_grads(gdn, x, C, dso=None):
    t = to_dev(x)
    o, st, saved = gdn.fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], chunk=C,
                           state_in=t["state_in"], out_dtype=t["dout"].dtype,
                           cu_seqlens_host=x["cu_seqlens"])
    return gdn.bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], saved, t["dout"],
                   chunk=C, state_in=t["state_in"],
                   dstate_out=None if dso is None else dso.cuda(),
                   cu_seqlens_host=x["cu_seqlens"])


def oracle_grads(x, dso=None):
    return oracle.bwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["g"]), f64(x["beta"]),
                      x["cu_seqlens"].numpy(), f64(x["dout"]), state_in=f64(x["state_in"]),
                      dstate_out=None if dso is None else f64(dso))


def dstate(x, seed):
    n = x["cu_seqlens"].numel() - 1
    hv, d = x["v"].shape[1], x["v"].shape[2]
    g = torch.Generator().manual_seed(seed)
    return torch.randn((n, hv, d, d), generator=g) / d


def check(gr, ref, tol):
    for name in NAMES:
        err = rel_err(gr[name], ref[name])
        assert err <= tol, (name, err)


def test_tiny_fp32_full_oracle(gdn):
    w = synth.workloads()["tiny"]
    x = synth.make_inputs(w.lengths, w.h_qk, w.h_v, w.d, dtype=w.dtype, seed=0, state_in=True,
                          dout=True, out_dtype=synth.F32)
    dso = dstate(x, 1)
    check(gpu_grads(gdn, x, w.chunk, dso), oracle_grads(x, dso), TOL[synth.F32])


@pytest.mark.parametrize("d,C", [(32, 16), (64, 32), (128, 64), (64, 64)])
@pytest.mark.parametrize("dtype", [synth.BF16, synth.F32])
def test_ragged_batches(gdn, d, C, dtype):
    lengths = [1, C - 1, C, C + 1, 3 * C + 5, 0, 2 * C]
    x = synth.make_inputs(lengths, 2, 4, d, dtype=dtype, seed=d + C + 1, state_in=True, dout=True,
                          out_dtype=synth.F32)
    dso = dstate(x, 2)
    check(gpu_grads(gdn, x, C, dso), oracle_grads(x, dso), TOL[dtype])


@pytest.mark.parametrize("dtype", [synth.BF16, synth.F32])
def test_slow_decay_and_no_final_gradient(gdn, dtype):
    """Slow decay makes the reverse boundary chain carry gradient across many chunks;
    dstate_out = NULL is treated as zero."""
    x = synth.make_inputs([400, 130], 2, 4, 64, dtype=dtype, seed=9, decay="slow", dout=True,
                          out_dtype=synth.F32)
    check(gpu_grads(gdn, x, 32), oracle_grads(x), TOL[dtype])


def test_bf16_upstream_gradient(gdn):
    """dO in bf16 (the output dtype of a bf16 forward)."""
    x = synth.make_inputs([150, 70], 2, 4, 64, dtype=synth.BF16, seed=10, dout=True)
    assert x["dout"].dtype == torch.bfloat16
    check(gpu_grads(gdn, x, 64), oracle_grads(x), 2e-3)


def test_deterministic(gdn):
    x = synth.make_inputs([300, 77, 64], 2, 4, 128, dtype=synth.BF16, seed=11, state_in=True,
                          dout=True)
    a = gpu_grads(gdn, x, 64)
    b = gpu_grads(gdn, x, 64)
    for name in NAMES:
        assert torch.equal(a[name], b[name]), name


def test_full_size_trainer_sampled(gdn):
    """The trainer workload (8 packed sequences, lengths U[512, 8192], 16/32 heads, d = 128,
    C = 64, bf16) in the benchmark's launch configuration; the oracle recomputes a seeded
    sample of (sequence, key head) groups of the shortest and of the longest sequence (the
    longest reverse chain)."""
    w = synth.workloads()["trainer"]
    x = synth.make_inputs(w.lengths, w.h_qk, w.h_v, w.d, dtype=w.dtype, seed=0, dout=True)
    gr = gpu_grads(gdn, x, w.chunk)
    for name in NAMES:
        assert torch.isfinite(gr[name]).all(), name
    cu = x["cu_seqlens"].tolist()
    grp = w.h_v // w.h_qk
    for s, hq in ((int(np.argmin(w.lengths)), 0), (int(np.argmin(w.lengths)), 11),
                  (int(np.argmax(w.lengths)), 6)):
        a, b = cu[s], cu[s + 1]
        hs = slice(hq * grp, (hq + 1) * grp)
        sub = {n: x[n][a:b, hq:hq + 1] for n in ("q", "k")}
        sub.update({n: x[n][a:b, hs] for n in ("v", "g", "beta", "dout")})
        ref = oracle.bwd(f64(sub["q"]), f64(sub["k"]), f64(sub["v"]), f64(sub["g"]),
                         f64(sub["beta"]), [0, b - a], f64(sub["dout"]))
        assert rel_err(gr["dq"][a:b, hq], ref["dq"][:, 0]) <= 2e-3
        assert rel_err(gr["dk"][a:b, hq], ref["dk"][:, 0]) <= 2e-3
        assert rel_err(gr["dv"][a:b, hs], ref["dv"]) <= 2e-3
        assert rel_err(gr["dg"][a:b, hs], ref["dg"]) <= 2e-3
        assert rel_err(gr["dbeta"][a:b, hs], ref["dbeta"]) <= 2e-3
        assert rel_err(gr["dstate_in"][s, hs], ref["dstate_in"][0]) <= 2e-3
