"""The token step's scaled state (S = c S~, the decay carried as the scalar c; the state made
explicit whenever c leaves [2^-64, 2^64]).  Strong decay drives c below 2^-64 every ~15
tokens, so the explicit step runs several times per chunk: every mode must still give the
same bits (prefill, decode, continued prefill), and the fp32 outputs must stay within the
oracle tolerance (the recurrence of the IsoExec page, section "Chunkwise-Parallel Recurrent
(CPR) Gated DeltaNet", in fp64)."""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_cpr_gb300 import synth
from helpers import f64, rel_err

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "g", "beta")


def strong_decay(x, seed):
    """g = -3 on about 80% of the tokens (c falls by e^-3 each), 0 on the rest."""
    gen = torch.Generator().manual_seed(seed)
    strong = torch.rand(x["g"].shape, generator=gen) < 0.8
    x["g"] = torch.where(strong, torch.full_like(x["g"], -3.0), torch.zeros_like(x["g"]))
    return x


@pytest.mark.parametrize("d,C,dtype", [(128, 64, synth.BF16), (64, 32, synth.F32), (32, 16, synth.BF16)])
def test_strong_decay_decode_equals_prefill(gdn, d, C, dtype):
    L0, M = 37, 90
    lengths = [L0 + M, L0 + M + 2]
    hqk, hv = 2, 4
    x = strong_decay(synth.make_inputs(lengths, hqk, hv, d, dtype=dtype, seed=d + C), seed=d)
    cu = x["cu_seqlens"].tolist()
    t = {n: x[n].cuda() for n in NAMES}
    o_full, s_full = gdn.prefill(t["q"], t["k"], t["v"], t["g"], t["beta"], x["cu_seqlens"].cuda(),
                                 chunk=C, out_dtype=torch.float32, cu_seqlens_host=x["cu_seqlens"])
    tdt = torch.bfloat16 if dtype == synth.BF16 else torch.float32
    cache = gdn.Cache(3, hqk, hv, d, C, dtype=tdt)
    slots = torch.tensor([2, 0], dtype=torch.int32, device="cuda")
    head = {n: torch.cat([x[n][cu[s]:cu[s] + L0] for s in range(2)]).cuda() for n in NAMES}
    cuh = synth.cu_seqlens_of([L0, L0])
    gdn.prefill(head["q"], head["k"], head["v"], head["g"], head["beta"], cuh.cuda(), chunk=C,
                out_dtype=torch.float32, cache=cache, slot_of_seq=slots, cu_seqlens_host=cuh)
    for i in range(M):
        tok = [cu[s] + L0 + i for s in range(2)]
        st = {n: x[n][tok].contiguous().cuda() for n in NAMES}
        od = gdn.decode_step(st["q"], st["k"], st["v"], st["g"], st["beta"], slots, cache,
                             out_dtype=torch.float32)
        for s in range(2):
            assert torch.equal(od[s], o_full[tok[s]]), (i, s)
    assert torch.equal(cache.running_state(2), s_full[0])
    c = cache.c_run[slots.long()]
    assert bool(((c >= 2.0 ** -64) & (c <= 2.0 ** 64)).all()), c
    if dtype == synth.F32:
        o_or, s_or, _ = oracle.fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["g"]), f64(x["beta"]),
                                   x["cu_seqlens"].numpy())
        assert rel_err(o_full, o_or) <= 1e-5
        assert rel_err(s_full, s_or) <= 1e-5


def test_strong_decay_continue_equals_prefill(gdn):
    """A continued prefill that resumes inside a chunk from a scaled running state."""
    hqk, hv, d, C = 2, 4, 128, 64
    P, L = [45, 70], [100, 30]
    total = [p + l for p, l in zip(P, L)]
    x = strong_decay(synth.make_inputs(total, hqk, hv, d, dtype=synth.BF16, seed=4), seed=5)
    cu = x["cu_seqlens"].tolist()
    t = {n: x[n].cuda() for n in NAMES}
    o_full, s_full = gdn.prefill(t["q"], t["k"], t["v"], t["g"], t["beta"], x["cu_seqlens"].cuda(),
                                 chunk=C, out_dtype=torch.float32, cu_seqlens_host=x["cu_seqlens"])
    cache = gdn.Cache(2, hqk, hv, d, C, dtype=torch.bfloat16)
    slots = torch.tensor([1, 0], dtype=torch.int32, device="cuda")
    head = {n: torch.cat([x[n][cu[s]:cu[s] + P[s]] for s in range(2)]).cuda() for n in NAMES}
    cuh = synth.cu_seqlens_of(P)
    gdn.prefill(head["q"], head["k"], head["v"], head["g"], head["beta"], cuh.cuda(), chunk=C,
                out_dtype=torch.float32, cache=cache, slot_of_seq=slots, cu_seqlens_host=cuh)
    tail = {n: torch.cat([x[n][cu[s] + P[s]:cu[s + 1]] for s in range(2)]).cuda() for n in NAMES}
    cut = synth.cu_seqlens_of(L)
    o_new, st_new = gdn.prefill_continue(tail["q"], tail["k"], tail["v"], tail["g"], tail["beta"], cut.cuda(),
                                         slots, cache, cu_seqlens_host=cut, out_dtype=torch.float32,
                                         want_state=True)
    cc = cut.tolist()
    for s in range(2):
        assert torch.equal(o_new[cc[s]:cc[s + 1]], o_full[cu[s] + P[s]:cu[s + 1]]), s
        assert torch.equal(st_new[s], s_full[s]), s
        assert torch.equal(cache.running_state(int(slots[s])), s_full[s]), s
