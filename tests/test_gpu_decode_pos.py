"""gdn_cpr_decode_step_pos: the decode step with the host's copy of the slot positions.

When no token of the step completes a chunk the resync kernels are not launched; the
results must be bit-identical to gdn_cpr_decode_step (checked step by step through chunk
boundaries, on the tensor-core and the SIMT boundary paths, and replayed from a CUDA graph).
A wrong claim (the host says no chunk completes, the cache says one does) is caught on the
device: the step changes nothing and the error word reads GDN_DEVERR_POS_HOST."""
import pytest
import torch

from gated_deltanet_cpr_gb300 import synth

pytestmark = pytest.mark.gpu

GDN_DEVERR_POS_HOST = 6


def prefilled_caches(gdn, lengths, hqk, hv, d, C, dtype, seed):
    x = synth.make_inputs(lengths, hqk, hv, d, dtype=dtype, seed=seed)
    t = {n: x[n].cuda() for n in ("q", "k", "v", "g", "beta")}
    caches = []
    for _ in range(2):
        cache = gdn.Cache(len(lengths), hqk, hv, d, C, dtype=t["q"].dtype)
        gdn.prefill(t["q"], t["k"], t["v"], t["g"], t["beta"], x["cu_seqlens"].cuda(), chunk=C, cache=cache,
                    cu_seqlens_host=x["cu_seqlens"])
        caches.append(cache)
    return caches


@pytest.mark.parametrize("d,C,dtype", [(128, 64, synth.BF16), (64, 32, synth.F32)])
def test_decode_pos_equals_decode(gdn, d, C, dtype):
    hqk, hv = 2, 4
    lengths = [C - 3, 2 * C - 1, C + 7]  # slot 1 completes a chunk on the first step
    a, b = prefilled_caches(gdn, lengths, hqk, hv, d, C, dtype, seed=71)
    slot = torch.tensor([2, 0, 1], dtype=torch.int32, device="cuda")
    pos = [lengths[2], lengths[0], lengths[1]]  # pos of slot[n]
    steps = C + 4
    z = synth.make_inputs([3 * steps], hqk, hv, d, dtype=dtype, seed=72)
    zt = {n: z[n].cuda() for n in ("q", "k", "v", "g", "beta")}
    for i in range(steps):
        sl = slice(3 * i, 3 * i + 3)
        args = (zt["q"][sl], zt["k"][sl], zt["v"][sl], zt["g"][sl], zt["beta"][sl], slot)
        oa = gdn.decode_step(*args, a, out_dtype=torch.float32)
        ob = gdn.decode_step(*args, b, out_dtype=torch.float32, pos_host=pos)
        assert torch.equal(oa, ob), i
        pos = [p + 1 for p in pos]
    for n in gdn.Cache.TENSORS:
        assert torch.equal(getattr(a, n), getattr(b, n)), n
    assert [int(p) for p in b.pos[slot.long()].cpu()] == pos


def test_wrong_host_positions_skip_the_step(gdn):
    hqk, hv, d, C = 2, 4, 128, 64
    cache, _ = prefilled_caches(gdn, [C - 1, 10], hqk, hv, d, C, synth.BF16, seed=73)
    slot = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    z = synth.make_inputs([2], hqk, hv, d, dtype=synth.BF16, seed=74)
    zt = {n: z[n].cuda() for n in ("q", "k", "v", "g", "beta")}
    before = {n: getattr(cache, n).clone() for n in gdn.Cache.TENSORS}
    shape = gdn.make_shape(2, 2, hqk, hv, d, C, torch.bfloat16, torch.float32)
    ws = gdn.alloc_workspace(gdn.workspace_bytes(shape, gdn.MODE_DECODE), "cuda")
    o = torch.full((2, hv, d), 7.0, device="cuda")
    # slot 0 sits at C - 1: its token completes a chunk, but the host claims position 5
    gdn.decode_step(zt["q"], zt["k"], zt["v"], zt["g"], zt["beta"], slot, cache, out_dtype=torch.float32,
                    ws=ws, o=o, pos_host=[5, 10])
    assert gdn.device_error(ws) == GDN_DEVERR_POS_HOST
    for n in gdn.Cache.TENSORS:
        assert torch.equal(getattr(cache, n), before[n]), n
    assert (o == 7.0).all()
    # the right positions run the step (with its resync)
    gdn.decode_step(zt["q"], zt["k"], zt["v"], zt["g"], zt["beta"], slot, cache, out_dtype=torch.float32,
                    ws=ws, o=o, pos_host=[C - 1, 10])
    assert gdn.device_error(ws) == 0
    assert cache.pos.tolist() == [C, 11]
    with pytest.raises(gdn.GdnError):
        gdn.decode_step(zt["q"], zt["k"], zt["v"], zt["g"], zt["beta"], slot, cache, pos_host=[-1, 11])


def test_decode_pos_graph_replay(gdn):
    """Steps with host positions captured in a CUDA graph (resync kernels absent except on the
    step that completes a chunk) replay to the bits of eager decode_step."""
    hqk, hv, d, C = 2, 4, 128, 64
    a, b = prefilled_caches(gdn, [C - 2, 3], hqk, hv, d, C, synth.BF16, seed=75)
    slot = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
    steps = 4
    z = synth.make_inputs([2 * steps], hqk, hv, d, dtype=synth.BF16, seed=76)
    zt = {n: z[n].cuda() for n in ("q", "k", "v", "g", "beta")}
    shape = gdn.make_shape(2, 2, hqk, hv, d, C, torch.bfloat16, torch.bfloat16)
    ws = gdn.alloc_workspace(gdn.workspace_bytes(shape, gdn.MODE_DECODE), "cuda")
    ob = torch.empty((steps, 2, hv, d), dtype=torch.bfloat16, device="cuda")
    start = {n: getattr(b, n).clone() for n in gdn.Cache.TENSORS}

    def run(i):
        sl = slice(2 * i, 2 * i + 2)
        gdn.decode_step(zt["q"][sl], zt["k"][sl], zt["v"][sl], zt["g"][sl], zt["beta"][sl], slot, b, ws=ws,
                        o=ob[i], pos_host=[C - 2 + i, 3 + i])

    run(0)  # first calls set up kernel attributes outside the capture
    for n in gdn.Cache.TENSORS:
        getattr(b, n).copy_(start[n])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(steps):
            run(i)
    g.replay()
    for i in range(steps):
        sl = slice(2 * i, 2 * i + 2)
        oa = gdn.decode_step(zt["q"][sl], zt["k"][sl], zt["v"][sl], zt["g"][sl], zt["beta"][sl], slot, a)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob[i]), i
    for n in gdn.Cache.TENSORS:
        assert torch.equal(getattr(a, n), getattr(b, n)), n
