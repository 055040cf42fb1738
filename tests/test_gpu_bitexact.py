"""Bit-equality across modes and batchings (the CPR contract: prefill, trainer forward and
decode give identical bits whatever the batch composition; IsoExec page, section
"Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet", and the per-region bitwise check
before registration described on the hegai.media page, section "Что именно объединяет
IsoExec").  These compare GPU against GPU with torch.equal."""
import numpy as np
import pytest
import torch

from gated_deltanet_cpr_gb300 import synth
from helpers import to_dev

pytestmark = pytest.mark.gpu


def prefill(gdn, x, C, cache=None, slot_of_seq=None, out=torch.float32):
    t = to_dev(x)
    return gdn.prefill(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], chunk=C,
                       state_in=t["state_in"], out_dtype=out, cache=cache,
                       slot_of_seq=slot_of_seq, cu_seqlens_host=x["cu_seqlens"])


def pack(seqs):
    """Concatenate per-sequence dicts (token tensors + optional state) into one batch."""
    out = {}
    for n in ("q", "k", "v", "g", "beta"):
        out[n] = torch.cat([s[n] for s in seqs])
    out["cu_seqlens"] = synth.cu_seqlens_of([s["q"].shape[0] for s in seqs])
    out["state_in"] = None if seqs[0]["state_in"] is None else torch.cat([s["state_in"] for s in seqs])
    return out


def split(x):
    cu = x["cu_seqlens"].tolist()
    res = []
    for s in range(len(cu) - 1):
        d = {n: x[n][cu[s]:cu[s + 1]] for n in ("q", "k", "v", "g", "beta")}
        d["state_in"] = None if x["state_in"] is None else x["state_in"][s:s + 1]
        res.append(d)
    return res


@pytest.mark.parametrize("dtype", [synth.BF16, synth.F32])
def test_prefill_equals_trainer_forward(gdn, dtype):
    x = synth.make_inputs([200, 64, 13], 2, 4, 64, dtype=dtype, seed=11, state_in=True)
    o1, s1 = prefill(gdn, x, 32)
    t = to_dev(x)
    o2, s2, _ = gdn.fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], chunk=32,
                        state_in=t["state_in"], out_dtype=torch.float32,
                        cu_seqlens_host=x["cu_seqlens"])
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_run_to_run_deterministic(gdn):
    x = synth.make_inputs([500, 77], 2, 4, 128, dtype=synth.BF16, seed=12)
    o1, s1 = prefill(gdn, x, 64)
    o2, s2 = prefill(gdn, x, 64)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_grouped_heads_equal_repeated_heads(gdn):
    x = synth.make_inputs([150, 40], 2, 4, 64, dtype=synth.BF16, seed=13)
    o1, s1 = prefill(gdn, x, 32)
    y = dict(x)
    rep = torch.arange(4) // 2
    y["q"], y["k"] = x["q"][:, rep].contiguous(), x["k"][:, rep].contiguous()
    o2, s2 = prefill(gdn, y, 32)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


@pytest.mark.parametrize("batch", [1, 7])
def test_batch_invariance_shuffled_packing(gdn, batch):
    """Sequences run alone, in batches of `batch`, and all together in a shuffled order
    give identical bits."""
    lengths = [int(v) for v in np.random.default_rng(14).integers(1, 400, size=14)]
    x = synth.make_inputs(lengths, 2, 4, 64, dtype=synth.BF16, seed=14, state_in=True)
    seqs = split(x)
    o_all, s_all = prefill(gdn, x, 64)
    cu = x["cu_seqlens"].tolist()
    perm = np.random.default_rng(1).permutation(len(seqs))
    for start in range(0, len(perm), batch):
        idx = perm[start:start + batch]
        xb = pack([seqs[i] for i in idx])
        ob, sb = prefill(gdn, xb, 64)
        cb = xb["cu_seqlens"].tolist()
        for j, i in enumerate(idx):
            assert torch.equal(ob[cb[j]:cb[j + 1]], o_all[cu[i]:cu[i + 1]]), i
            assert torch.equal(sb[j], s_all[i]), i


@pytest.mark.parametrize("L0,M,C", [(0, 70, 32), (64, 64, 64), (50, 100, 64), (33, 40, 16),
                                    (128, 1, 64), (1, 130, 32)])
def test_decode_equals_prefill(gdn, L0, M, C):
    """Prefill L0 tokens into a cache, decode M more one by one: every decode output and the
    final running state equal a single prefill of all L0 + M tokens, bit for bit."""
    lengths = [L0 + M, L0 + M + 3]
    x = synth.make_inputs(lengths, 2, 4, 64, dtype=synth.BF16, seed=L0 + M + C, state_in=True)
    o_full, s_full = prefill(gdn, x, C)
    seqs = split(x)
    head = pack([{n: (s[n][:L0] if n != "state_in" else s[n]) for n in s} for s in seqs])
    slots = torch.tensor([3, 1], dtype=torch.int32, device="cuda")
    cache = gdn.Cache(5, 2, 4, 64, C, dtype=torch.bfloat16)
    prefill(gdn, head, C, cache=cache, slot_of_seq=slots)
    cu = x["cu_seqlens"].tolist()
    for i in range(M):
        tok = [cu[s] + L0 + i for s in range(2)]
        st = {n: x[n][tok].contiguous().cuda() for n in ("q", "k", "v", "g", "beta")}
        od = gdn.decode_step(st["q"], st["k"], st["v"], st["g"], st["beta"], slots, cache,
                             out_dtype=torch.float32)
        for s in range(2):
            assert torch.equal(od[s], o_full[tok[s]]), (i, s)
    assert torch.equal(cache.pos[slots.long()].cpu(), torch.tensor([L0 + M] * 2, dtype=torch.int32))
    # the second sequence still has 3 prefill tokens left: finish them by decode too
    for i in range(M, M + 3):
        tok = [cu[1] + L0 + i]
        st = {n: x[n][tok].contiguous().cuda() for n in ("q", "k", "v", "g", "beta")}
        od = gdn.decode_step(st["q"], st["k"], st["v"], st["g"], st["beta"], slots[1:], cache,
                             out_dtype=torch.float32)
        assert torch.equal(od[0], o_full[tok[0]])
    assert torch.equal(cache.running_state(3), s_full[0])
    assert torch.equal(cache.running_state(1), s_full[1])


def test_decode_checkpoint_resume(gdn):
    """Copy the cache to the host mid-decode, scramble the device copy, restore it and
    continue: the bits are unchanged (the cache is the full resumable state)."""
    C = 32
    x = synth.make_inputs([90], 2, 4, 64, dtype=synth.BF16, seed=21)
    o_full, s_full = prefill(gdn, x, C)
    L0 = 20
    cache = gdn.Cache(1, 2, 4, 64, C, dtype=torch.bfloat16)
    head = {n: x[n][:L0] for n in ("q", "k", "v", "g", "beta")}
    head["state_in"] = None
    head["cu_seqlens"] = synth.cu_seqlens_of([L0])
    prefill(gdn, head, C, cache=cache)
    slot = torch.zeros(1, dtype=torch.int32, device="cuda")
    for i in range(L0, 90):
        if i == 50:
            saved = cache.state_dict()
            for n in cache.TENSORS:
                getattr(cache, n).zero_()
            cache.load_state_dict(saved)
        st = {n: x[n][i:i + 1].cuda() for n in ("q", "k", "v", "g", "beta")}
        od = gdn.decode_step(st["q"], st["k"], st["v"], st["g"], st["beta"], slot, cache,
                             out_dtype=torch.float32)
        assert torch.equal(od[0], o_full[i])
    assert torch.equal(cache.running_state(0), s_full[0])


def test_device_errors_are_reported_not_faulted(gdn):
    x = synth.make_inputs([40, 30], 2, 4, 64, dtype=synth.BF16, seed=22)
    t = to_dev(x)
    # device cu_seqlens disagree with the host copy -> error word, no work, no fault
    bad = torch.tensor([0, 35, 70], dtype=torch.int32, device="cuda")
    ws = gdn.alloc_workspace(1 << 24, "cuda")
    gdn.prefill(t["q"], t["k"], t["v"], t["g"], t["beta"], bad, chunk=32,
                cu_seqlens_host=x["cu_seqlens"], ws=ws)
    assert gdn.device_error(ws) == 1
    # slot out of range in decode
    cache = gdn.Cache(2, 2, 4, 64, 32, dtype=torch.bfloat16)
    slot = torch.tensor([5], dtype=torch.int32, device="cuda")
    ws2 = gdn.alloc_workspace(1 << 24, "cuda")
    st = {n: x[n][:1].cuda() for n in ("q", "k", "v", "g", "beta")}
    gdn.decode_step(st["q"], st["k"], st["v"], st["g"], st["beta"], slot, cache, ws=ws2)
    assert gdn.device_error(ws2) == 2
    # the context is still usable
    o, _ = gdn.prefill(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], chunk=32,
                       cu_seqlens_host=x["cu_seqlens"], ws=ws)
    assert gdn.device_error(ws) == 0
    assert torch.isfinite(o.float()).all()


@pytest.mark.parametrize("L0,M", [(64, 64), (100, 90), (0, 130)])
def test_decode_equals_prefill_tensor_core_boundary(gdn, L0, M):
    """d = 128, C = 64, bf16: the shape whose boundary pass runs on tcgen05 tensor cores in
    both prefill and decode resynchronisation; decode must still equal prefill bit for bit."""
    C, d = 64, 128
    lengths = [L0 + M, L0 + M + 5, 3]
    x = synth.make_inputs(lengths, 2, 4, d, dtype=synth.BF16, seed=L0 + 7 * M, state_in=True,
                          decay="slow")
    o_full, s_full = prefill(gdn, x, C)
    seqs = split(x)
    head = pack([{n: (s[n][:min(L0, s["q"].shape[0])] if n != "state_in" else s[n]) for n in s}
                 for s in seqs[:2]])
    slots = torch.tensor([1, 0], dtype=torch.int32, device="cuda")
    cache = gdn.Cache(2, 2, 4, d, C, dtype=torch.bfloat16)
    prefill(gdn, head, C, cache=cache, slot_of_seq=slots)
    cu = x["cu_seqlens"].tolist()
    for i in range(M):
        tok = [cu[s] + L0 + i for s in range(2)]
        st = {n: x[n][tok].contiguous().cuda() for n in ("q", "k", "v", "g", "beta")}
        od = gdn.decode_step(st["q"], st["k"], st["v"], st["g"], st["beta"], slots, cache,
                             out_dtype=torch.float32)
        for s in range(2):
            assert torch.equal(od[s], o_full[tok[s]]), (i, s)
    assert torch.equal(cache.running_state(1), s_full[0])
