"""Oracle parity of the tensor-core boundary path where boundary states carry memory.

Under the default decay g = -softplus(N(0,1)) a chunk of 64 tokens multiplies the state by
about e^-45, so S^(j) holds only the last few tokens of chunk j-1 and any error in the
chained term gamma_C S^(j-1) is invisible.  These cases run the shape that takes the
tcgen05 path (d = 128, C = 64, bf16 inputs, 16 query/key heads shared by 32 value heads)
under slow decay (g = -0.02 sigmoid(N(0,1)), about e^-0.64 per chunk) and without decay
(g = 0, where only the delta rule's projection forgets), over chains of 32 to 512 chunk
steps, and compare o, the final state, every saved boundary state S^(j) and all six
gradients with the fp64 oracle (the token recurrence of the IsoExec page, section
"Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet").

Tolerance: max|GPU - oracle| / max|oracle| per tensor <= 2e-3 (bf16 inputs).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_cpr_gb300 import synth
from helpers import f64, oracle_full, oracle_pairs, rel_err, to_dev

pytestmark = pytest.mark.gpu

TOL = 2e-3
HQK, HV, D, C = 16, 32, 128, 64
GRADS = ("dq", "dk", "dv", "dg", "dbeta", "dstate_in")


def gpu_fwd(gdn, x):
    t = to_dev(x)
    return gdn.fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], chunk=C,
                   state_in=t["state_in"], out_dtype=torch.float32,
                   cu_seqlens_host=x["cu_seqlens"])


@pytest.mark.parametrize("decay", ["slow", "none"])
def test_chained_boundaries_all_heads(gdn, decay):
    """Two sequences of 2085 and 2048 tokens (33 and 32 chained chunk steps, one ragged
    tail), every head: o, state_out and every S^(j) against the oracle."""
    lengths = [2085, 2048]
    x = synth.make_inputs(lengths, HQK, HV, D, dtype=synth.BF16, seed=21, decay=decay,
                          state_in=True)
    o, st, bnd = gpu_fwd(gdn, x)
    o_ref, st_ref, bnd_ref = oracle_full(x, chunk=C)
    assert bnd.shape[0] == bnd_ref.shape[0] == 33 + 32
    e = (rel_err(o, o_ref), rel_err(st, st_ref), rel_err(bnd, bnd_ref))
    assert max(e) <= TOL, e
    # the last boundary state of each sequence carries the whole chain
    for s, j in ((0, 32), (1, 31 + 33)):
        assert rel_err(bnd[j], bnd_ref[j]) <= TOL, (s, j)


def test_long_context_chain_sampled_pairs(gdn):
    """The longest sequence of the long-context workload (32713 tokens: 511 chained chunk
    steps and a tail) under slow decay, all 32 heads on the GPU; the oracle recomputes a
    seeded sample of heads one by one: o, the final state and every S^(j)."""
    L = max(synth.workloads()["longctx"].lengths)
    assert L >= 16384
    x = synth.make_inputs([L], HQK, HV, D, dtype=synth.BF16, seed=22, decay="slow")
    o, st, bnd = gpu_fwd(gdn, x)
    assert bnd.shape[0] == (L + C - 1) // C
    rng = np.random.default_rng(22)
    heads = sorted(set(int(h) for h in rng.integers(0, HV, 3)))
    ref = oracle_pairs(x, [(0, h) for h in heads], chunk=C)
    for (_, h), (o_ref, st_ref, bnd_ref) in ref.items():
        assert rel_err(o[:, h], o_ref) <= TOL, h
        assert rel_err(st[0, h], st_ref) <= TOL, h
        assert rel_err(bnd[:, h], bnd_ref) <= TOL, h


def _grads(gdn, x, dso=None):
    t = to_dev(x)
    _, _, saved = gpu_fwd(gdn, x)
    return gdn.bwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], saved, t["dout"],
                   chunk=C, state_in=t["state_in"],
                   dstate_out=None if dso is None else dso.cuda(),
                   cu_seqlens_host=x["cu_seqlens"])


@pytest.mark.parametrize("decay", ["slow", "none"])
def test_backward_chained_gradients(gdn, decay):
    """Backward on the tensor-core path with the reverse chain carrying gradient over 17
    and 16 chunk steps (1100 and 1024 tokens), state_in and dstate_out given: all six
    gradients against the oracle's reverse recurrence."""
    lengths = [1100, 1024]
    x = synth.make_inputs(lengths, 2, 4, D, dtype=synth.BF16, seed=23, decay=decay,
                          state_in=True, dout=True, out_dtype=synth.F32)
    gen = torch.Generator().manual_seed(24)
    dso = torch.randn((2, 4, D, D), generator=gen) / D
    gr = _grads(gdn, x, dso)
    ref = oracle.bwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["g"]), f64(x["beta"]),
                     x["cu_seqlens"].numpy(), f64(x["dout"]), state_in=f64(x["state_in"]),
                     dstate_out=f64(dso))
    errs = {n: rel_err(gr[n], ref[n]) for n in GRADS}
    assert max(errs.values()) <= TOL, errs


def test_backward_grouped_heads_long_chain(gdn):
    """The full 16/32-head shape under slow decay on one 4096-token sequence (64 reverse
    chain steps); the oracle recomputes two key-head groups (their two value heads each)."""
    x = synth.make_inputs([4096], HQK, HV, D, dtype=synth.BF16, seed=25, decay="slow",
                          dout=True)
    gr = _grads(gdn, x)
    grp = HV // HQK
    for hq in (3, 14):
        hs = slice(hq * grp, (hq + 1) * grp)
        ref = oracle.bwd(f64(x["q"][:, hq:hq + 1]), f64(x["k"][:, hq:hq + 1]), f64(x["v"][:, hs]),
                         f64(x["g"][:, hs]), f64(x["beta"][:, hs]), [0, 4096],
                         f64(x["dout"][:, hs]))
        errs = {"dq": rel_err(gr["dq"][:, hq], ref["dq"][:, 0]),
                "dk": rel_err(gr["dk"][:, hq], ref["dk"][:, 0]),
                "dv": rel_err(gr["dv"][:, hs], ref["dv"]),
                "dg": rel_err(gr["dg"][:, hs], ref["dg"]),
                "dbeta": rel_err(gr["dbeta"][:, hs], ref["dbeta"]),
                "dstate_in": rel_err(gr["dstate_in"][0, hs], ref["dstate_in"][0])}
        assert max(errs.values()) <= TOL, (hq, errs)
