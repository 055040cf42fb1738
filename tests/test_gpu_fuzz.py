"""Seeded sweep over the supported configuration space, each case against the fp64 oracle and
for decode == prefill bit equality.

Every case draws d in {32, 64, 128}, C in {16, 32, 64}, bf16 or fp32 inputs, 1 or 2
query/key heads with 1 or 2 value heads per group, default or slow decay, an optional
state_in, and 1-5 sequences of ragged lengths in [0, 5C] (empty ones included).  It checks
prefill o and state_out and all six gradients of fwd + bwd against the oracle (2e-3 for bf16,
1e-5 for fp32, max|d|/max|ref| per tensor), then prefills the first sequence up to a random
split point into a cache and decodes the rest token by token (host positions on every other
step), which must reproduce the prefill's outputs and final state bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_cpr_gb300 import synth
from helpers import f64, oracle_full, rel_err, to_dev

pytestmark = pytest.mark.gpu

TOL = {synth.F32: 1e-5, synth.BF16: 2e-3}


def draw(rng):
    if rng.random() < 0.35:  # the tensor-core boundary path's shape
        d, C, dtype = 128, 64, synth.BF16
    else:
        d = int(rng.choice([32, 64, 128]))
        C = int(rng.choice([16, 32, 64]))
        dtype = synth.BF16 if rng.random() < 0.6 else synth.F32
    hqk = int(rng.choice([1, 2]))
    hv = hqk * int(rng.choice([1, 2]))
    n = int(rng.integers(1, 6))
    lengths = [int(rng.integers(0, 5 * C + 1)) for _ in range(n)]
    if lengths[0] < 2:
        lengths[0] = int(rng.integers(2, 5 * C + 1))
    if n > 1 and rng.random() < 0.3:
        lengths[int(rng.integers(1, n))] = 0
    decay = "slow" if rng.random() < 0.4 else "default"
    return d, C, dtype, hqk, hv, lengths, decay, bool(rng.random() < 0.5)


@pytest.mark.parametrize("case", range(48))
def test_fuzz_case(gdn, case):
    rng = np.random.default_rng(1000 + case)
    d, C, dtype, hqk, hv, lengths, decay, with_state = draw(rng)
    x = synth.make_inputs(lengths, hqk, hv, d, dtype=dtype, seed=2000 + case, decay=decay,
                          state_in=with_state, dout=True, out_dtype=synth.F32)
    t = to_dev(x)
    desc = (d, C, dtype, hqk, hv, lengths, decay, with_state)
    # prefill against the oracle
    o, st = gdn.prefill(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], chunk=C,
                        state_in=t["state_in"], out_dtype=torch.float32, cu_seqlens_host=x["cu_seqlens"])
    o_ref, st_ref, _ = oracle_full(x)
    if sum(lengths):
        assert rel_err(o, o_ref) <= TOL[dtype], desc
    assert rel_err(st, st_ref) <= TOL[dtype], desc
    # trainer forward + backward against the oracle
    o2, st2, saved = gdn.fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], chunk=C,
                             state_in=t["state_in"], out_dtype=torch.float32, cu_seqlens_host=x["cu_seqlens"])
    assert torch.equal(o2, o) and torch.equal(st2, st), desc
    gr = gdn.bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], saved, t["dout"], chunk=C,
                 state_in=t["state_in"], cu_seqlens_host=x["cu_seqlens"])
    ref = oracle.bwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["g"]), f64(x["beta"]),
                     x["cu_seqlens"].numpy(), f64(x["dout"]), state_in=f64(x["state_in"]))
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dstate_in"):
        if name != "dstate_in" and not sum(lengths):
            continue
        assert rel_err(gr[name], ref[name]) <= TOL[dtype], (name, desc)
    # decode the first sequence from a random split point: bits equal the prefill's
    L0 = lengths[0]
    split = int(rng.integers(0, L0))
    cache = gdn.Cache(2, hqk, hv, d, C, dtype=t["q"].dtype)
    slot = torch.tensor([1], dtype=torch.int32, device="cuda")
    cu_head = torch.tensor([0, split], dtype=torch.int32)
    sin = None if t["state_in"] is None else t["state_in"][:1].contiguous()
    gdn.prefill(t["q"][:split], t["k"][:split], t["v"][:split], t["g"][:split], t["beta"][:split],
                cu_head.cuda(), chunk=C, state_in=sin, out_dtype=torch.float32, cache=cache,
                slot_of_seq=slot, cu_seqlens_host=cu_head)
    for i in range(split, L0):
        sl = slice(i, i + 1)
        od = gdn.decode_step(t["q"][sl], t["k"][sl], t["v"][sl], t["g"][sl], t["beta"][sl], slot, cache,
                             out_dtype=torch.float32, pos_host=[i] if i % 2 else None)
        assert torch.equal(od[0], o[i]), (i, desc)
    assert torch.equal(cache.running_state([1])[0], st[0]), desc
