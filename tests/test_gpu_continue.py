"""Prefill continued from a decode cache (gdn_cpr_prefill_continue): chunked prefill and
multi-token decode.  The contract is the CPR one (IsoExec page, section "Chunkwise-Parallel
Recurrent (CPR) Gated DeltaNet"): extending a cached sequence gives the bits of one
prefill of the whole sequence, whatever the split points, and the cache it leaves behind
decodes on bit-identically.  Compared GPU against GPU with torch.equal, plus one fp64
oracle check of the continued outputs.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_deltanet_cpr_gb300 import synth
from helpers import f64, rel_err

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "g", "beta")


def seq_slices(x):
    cu = x["cu_seqlens"].tolist()
    return [{n: x[n][cu[s]:cu[s + 1]] for n in NAMES} for s in range(len(cu) - 1)]


def packed(parts, dev="cuda"):
    out = {n: torch.cat([p[n] for p in parts]).to(dev) for n in NAMES}
    return out, synth.cu_seqlens_of([p["q"].shape[0] for p in parts])


def full_prefill(gdn, seqs, hqk, hv, d, C, dtype, slots_n):
    x, cu = packed(seqs)
    cache = gdn.Cache(slots_n, hqk, hv, d, C, dtype=dtype)
    slots = torch.arange(len(seqs), dtype=torch.int32, device="cuda")
    o, st = gdn.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], cu.cuda(), chunk=C,
                        cu_seqlens_host=cu, out_dtype=torch.float32, cache=cache, slot_of_seq=slots)
    return o, st, cache, cu.tolist()


def cut(seqs, a, b):
    """Tokens [a[i], b[i]) of every sequence."""
    return [{n: s[n][a[i]:b[i]] for n in NAMES} for i, s in enumerate(seqs)]


def same_cache(cache_a, slot_a, cache_b, slot_b, pos, C):
    assert torch.equal(cache_a.s_run[slot_a], cache_b.s_run[slot_b])
    assert torch.equal(cache_a.c_run[slot_a], cache_b.c_run[slot_b])
    assert torch.equal(cache_a.s_bnd[slot_a], cache_b.s_bnd[slot_b])
    assert int(cache_a.pos[slot_a]) == int(cache_b.pos[slot_b]) == pos
    r = pos % C
    for n in ("tail_k", "tail_v", "tail_g", "tail_beta"):
        assert torch.equal(getattr(cache_a, n)[slot_a, :r], getattr(cache_b, n)[slot_b, :r]), n


CASES = [
    # (dtype, d, C, prefix lengths, continuation lengths)
    (synth.BF16, 128, 64, [0, 1, 63, 64, 65, 130, 200], [5, 0, 64, 1, 130, 7, 300]),
    (synth.F32, 64, 32, [3, 32, 50, 0], [40, 1, 96, 33]),
    (synth.BF16, 32, 16, [17, 16, 5], [2, 40, 11]),
]


@pytest.mark.parametrize("dtype,d,C,P,L", CASES)
def test_continue_equals_single_prefill(gdn, dtype, d, C, P, L):
    hqk, hv = 2, 4
    total = [p + l for p, l in zip(P, L)]
    x = synth.make_inputs(total, hqk, hv, d, dtype=dtype, seed=d + C)
    seqs = seq_slices(x)
    tdt = torch.bfloat16 if dtype == synth.BF16 else torch.float32
    n = len(seqs)
    o_ref, st_ref, cache_ref, cu_ref = full_prefill(gdn, seqs, hqk, hv, d, C, tdt, n)
    # prefix into a second cache, slots reversed, then continue
    cache = gdn.Cache(n + 2, hqk, hv, d, C, dtype=tdt)
    slots = torch.tensor([n + 1 - i for i in range(n)], dtype=torch.int32, device="cuda")
    xp, cup = packed(cut(seqs, [0] * n, P))
    gdn.prefill(xp["q"], xp["k"], xp["v"], xp["g"], xp["beta"], cup.cuda(), chunk=C,
                cu_seqlens_host=cup, out_dtype=torch.float32, cache=cache, slot_of_seq=slots)
    xc, cuc = packed(cut(seqs, P, total))
    o_new, st_new = gdn.prefill_continue(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], cuc.cuda(),
                                         slots, cache, pos_host=P, cu_seqlens_host=cuc,
                                         out_dtype=torch.float32, want_state=True)
    cc = cuc.tolist()
    for i in range(n):
        assert torch.equal(o_new[cc[i]:cc[i + 1]], o_ref[cu_ref[i] + P[i]:cu_ref[i + 1]]), i
        assert torch.equal(st_new[i], st_ref[i]), i
        same_cache(cache_ref, i, cache, int(slots[i]), total[i], C)
    if dtype == synth.F32:  # the continued outputs against the fp64 recurrence of the whole sequences
        o_or, _, _ = oracle.fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["g"]), f64(x["beta"]),
                                x["cu_seqlens"].numpy())
        cx = x["cu_seqlens"].tolist()
        ref = np.concatenate([o_or[cx[i] + P[i]:cx[i + 1]] for i in range(n)])
        assert rel_err(o_new, ref) <= 1e-5


def test_multi_token_decode_steps(gdn):
    """Several short continuations in a row (1, 3, 7, 64, 2, 0, 61 tokens) equal one prefill."""
    hqk, hv, d, C = 2, 4, 128, 64
    steps = [1, 3, 7, 64, 2, 0, 61]
    P = [100, 64]
    total = [p + sum(steps) for p in P]
    x = synth.make_inputs(total, hqk, hv, d, dtype=synth.BF16, seed=5)
    seqs = seq_slices(x)
    o_ref, st_ref, cache_ref, cu_ref = full_prefill(gdn, seqs, hqk, hv, d, C, torch.bfloat16, 2)
    cache = gdn.Cache(2, hqk, hv, d, C, dtype=torch.bfloat16)
    slots = torch.tensor([1, 0], dtype=torch.int32, device="cuda")
    xp, cup = packed(cut(seqs, [0, 0], P))
    gdn.prefill(xp["q"], xp["k"], xp["v"], xp["g"], xp["beta"], cup.cuda(), chunk=C,
                cu_seqlens_host=cup, out_dtype=torch.float32, cache=cache, slot_of_seq=slots)
    at = list(P)
    for L in steps:
        xc, cuc = packed(cut(seqs, at, [a + L for a in at]))
        o_new, _ = gdn.prefill_continue(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], cuc.cuda(),
                                        slots, cache, cu_seqlens_host=cuc, out_dtype=torch.float32)
        cc = cuc.tolist()
        for i in range(2):
            assert torch.equal(o_new[cc[i]:cc[i + 1]], o_ref[cu_ref[i] + at[i]:cu_ref[i] + at[i] + L])
        at = [a + L for a in at]
    for i in range(2):
        same_cache(cache_ref, i, cache, int(slots[i]), total[i], C)


def test_continue_between_decode_steps(gdn):
    """prefill -> 3 decode steps -> continue by 70 -> 2 decode steps: every output and the
    final cache equal one prefill of the whole sequences."""
    hqk, hv, d, C = 2, 4, 128, 64
    P, L = [61, 128], 70
    total = [p + 3 + L + 2 for p in P]
    x = synth.make_inputs(total, hqk, hv, d, dtype=synth.BF16, seed=8)
    seqs = seq_slices(x)
    o_ref, _, cache_ref, cu_ref = full_prefill(gdn, seqs, hqk, hv, d, C, torch.bfloat16, 2)
    cache = gdn.Cache(2, hqk, hv, d, C, dtype=torch.bfloat16)
    slots = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    xp, cup = packed(cut(seqs, [0, 0], P))
    gdn.prefill(xp["q"], xp["k"], xp["v"], xp["g"], xp["beta"], cup.cuda(), chunk=C,
                cu_seqlens_host=cup, out_dtype=torch.float32, cache=cache, slot_of_seq=slots)
    at = list(P)

    def decode():
        tok = {n: torch.stack([seqs[i][n][at[i]] for i in range(2)]).cuda() for n in NAMES}
        od = gdn.decode_step(tok["q"], tok["k"], tok["v"], tok["g"], tok["beta"], slots, cache,
                             out_dtype=torch.float32)
        for i in range(2):
            assert torch.equal(od[i], o_ref[cu_ref[i] + at[i]])
            at[i] += 1

    for _ in range(3):
        decode()
    xc, cuc = packed(cut(seqs, at, [a + L for a in at]))
    o_new, _ = gdn.prefill_continue(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], cuc.cuda(), slots,
                                    cache, cu_seqlens_host=cuc, out_dtype=torch.float32)
    cc = cuc.tolist()
    for i in range(2):
        assert torch.equal(o_new[cc[i]:cc[i + 1]], o_ref[cu_ref[i] + at[i]:cu_ref[i] + at[i] + L])
    at = [a + L for a in at]
    for _ in range(2):
        decode()
    for i in range(2):
        same_cache(cache_ref, i, cache, int(slots[i]), total[i], C)


def test_position_mismatch_is_a_device_error(gdn):
    """A host position that disagrees with the cache is caught on the device (work-list
    check): nothing runs, the cache is untouched and the error word says cu_seqlens."""
    hqk, hv, d, C = 2, 4, 64, 32
    x = synth.make_inputs([40, 9], hqk, hv, d, dtype=synth.BF16, seed=3)
    seqs = seq_slices(x)
    cache = gdn.Cache(2, hqk, hv, d, C, dtype=torch.bfloat16)
    slots = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    xp, cup = packed(cut(seqs, [0, 0], [30, 4]))
    gdn.prefill(xp["q"], xp["k"], xp["v"], xp["g"], xp["beta"], cup.cuda(), chunk=C,
                cu_seqlens_host=cup, out_dtype=torch.float32, cache=cache, slot_of_seq=slots)
    before = {n: getattr(cache, n).clone() for n in gdn.Cache.TENSORS}
    xc, cuc = packed(cut(seqs, [30, 4], [40, 9]))
    shape = gdn.make_shape(2, 15, hqk, hv, d, C, torch.bfloat16, torch.float32)
    ws = gdn.alloc_workspace(gdn.workspace_bytes(shape, gdn.MODE_CONTINUE, cuc), "cuda")
    gdn.prefill_continue(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], cuc.cuda(), slots, cache,
                         pos_host=[30, 5], cu_seqlens_host=cuc, out_dtype=torch.float32, ws=ws)
    assert gdn.device_error(ws) == 1  # GDN_DEVERR_CU_SEQLENS
    for n in gdn.Cache.TENSORS:
        assert torch.equal(getattr(cache, n), before[n]), n
