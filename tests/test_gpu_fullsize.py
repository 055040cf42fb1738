"""Full-size bit-equality on the long-context and decode workloads.

- Long context: 64 sequences with lengths log-uniform in [128, 32768] (about 3.8e5 tokens),
  16/32 heads, d = 128, C = 64, bf16, prefilled in batches of 1, 7 and 64 with the packing
  order shuffled (seed 1): every sequence's o and final state are bit-identical, and the
  longest sequence matches the fp64 oracle on sampled heads.
- Decode: 256 sequences prefilled with 2048 tokens, then 128 decode steps with a
  resynchronisation every 64 tokens: every decode output and the final running states
  equal a single prefill of all 2176 tokens, bit for bit.
Inputs are generated on the CPU from their seeds, sequence by sequence, so that any packing
sees identical per-sequence values.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_cpr_gb300 import synth
from helpers import oracle_pairs, rel_err

pytestmark = pytest.mark.gpu


def per_sequence_inputs(lengths, hqk, hv, d, seed):
    return [synth.make_inputs([L], hqk, hv, d, dtype=synth.BF16, seed=seed + 17 * i)
            for i, L in enumerate(lengths)]


def pack(seqs, idx, dev="cuda"):
    out = {n: torch.cat([seqs[i][n] for i in idx]).to(dev) for n in ("q", "k", "v", "g", "beta")}
    cu = synth.cu_seqlens_of([seqs[i]["q"].shape[0] for i in idx])
    return out, cu


def run(gdn, x, cu, C=64, cache=None, slot_of_seq=None):
    return gdn.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], cu.cuda(), chunk=C,
                       cu_seqlens_host=cu, out_dtype=torch.bfloat16, cache=cache,
                       slot_of_seq=slot_of_seq)


def test_long_context_batch_invariance(gdn):
    w = synth.workloads()["longctx"]
    seqs = per_sequence_inputs(w.lengths, w.h_qk, w.h_v, w.d, seed=0)
    perm = np.random.default_rng(1).permutation(len(seqs))
    results = {}
    for batch in (64, 7, 1):
        outs, states = {}, {}
        for start in range(0, len(perm), batch):
            idx = [int(i) for i in perm[start:start + batch]]
            x, cu = pack(seqs, idx)
            o, st = run(gdn, x, cu)
            c = cu.tolist()
            for j, i in enumerate(idx):
                outs[i] = o[c[j]:c[j + 1]].clone()
                states[i] = st[j].clone()
            del x, o, st
        results[batch] = (outs, states)
    ref_o, ref_s = results[64]
    for batch in (7, 1):
        o_b, s_b = results[batch]
        for i in range(len(seqs)):
            assert torch.equal(o_b[i], ref_o[i]), (batch, i)
            assert torch.equal(s_b[i], ref_s[i]), (batch, i)
    assert all(torch.isfinite(ref_o[i].float()).all() for i in range(len(seqs)))
    # the longest sequence (511 chained chunk steps) against the fp64 oracle on sampled
    # heads, from an fp32-output run whose RNE is the batched bf16 output
    i = int(np.argmax(w.lengths))
    x, cu = pack(seqs, [i])
    o32, st32 = gdn.prefill(x["q"], x["k"], x["v"], x["g"], x["beta"], cu.cuda(), chunk=64,
                            cu_seqlens_host=cu, out_dtype=torch.float32)
    assert torch.equal(o32.to(torch.bfloat16), ref_o[i])
    assert torch.equal(st32[0], ref_s[i])
    for (_, h), (o_ref, st_ref, _) in oracle_pairs(seqs[i], [(0, 5), (0, 30)]).items():
        assert rel_err(o32[:, h], o_ref) <= 2e-3, h
        assert rel_err(st32[0, h], st_ref) <= 2e-3, h


def test_decode_workload_equals_prefill(gdn):
    w = synth.workloads()["decode"]
    N, L0, M = len(w.lengths), w.lengths[0], w.decode_steps
    x = synth.make_inputs([L0 + M] * N, w.h_qk, w.h_v, w.d, dtype=synth.BF16, seed=0)
    dev = {n: x[n].cuda() for n in ("q", "k", "v", "g", "beta")}
    o_full, s_full = run(gdn, dev, x["cu_seqlens"])
    # prefill the first 2048 tokens of every sequence into a cache (slots reversed)
    cu = x["cu_seqlens"].tolist()
    head_idx = torch.cat([torch.arange(cu[s], cu[s] + L0) for s in range(N)]).cuda()
    head = {n: dev[n].index_select(0, head_idx).contiguous() for n in dev}
    cu_head = synth.cu_seqlens_of([L0] * N)
    slots = torch.arange(N - 1, -1, -1, dtype=torch.int32, device="cuda")
    cache = gdn.Cache(N, w.h_qk, w.h_v, w.d, w.chunk, dtype=torch.bfloat16)
    run(gdn, head, cu_head, cache=cache, slot_of_seq=slots)
    starts = torch.tensor(cu[:-1], device="cuda")
    for i in range(M):
        tok = starts + L0 + i
        st = {n: dev[n].index_select(0, tok).contiguous() for n in dev}
        od = gdn.decode_step(st["q"], st["k"], st["v"], st["g"], st["beta"], slots, cache,
                             out_dtype=torch.bfloat16)
        assert torch.equal(od, o_full.index_select(0, tok)), i
    assert torch.equal(cache.running_state(slots.long()), s_full)
    assert torch.equal(cache.pos.cpu(), torch.full((N,), L0 + M, dtype=torch.int32))
