"""The decode step for callers that cannot allocate device memory.

gdn_cpr_decode_step_noalloc runs the ordinary decode step with its workspace placed in a
fixed device array inside the library (for serving loops whose device memory is reserved
up front, or hosts without a device allocator).  This checks, through the C ABI, that two
calls in a row give the same outputs and cache contents as the ordinary entry point with
a caller-provided workspace -- including steps where a slot completes a chunk and the
resynchronisation runs in the built-in scratch -- and that requests larger than the
array are refused.  Kept in its own file, collected last, so that a failure here leaves
every other test already run.
"""
import ctypes

import pytest
import torch

from gated_deltanet_cpr_gb300 import synth
from helpers import rel_err

pytestmark = pytest.mark.gpu


def make_cache(gdn, slots, hqk, hv, d, C, positions, seed):
    cache = gdn.Cache(slots, hqk, hv, d, C, dtype=torch.bfloat16)
    gen = torch.Generator(device="cuda").manual_seed(seed)
    cache.s_run.normal_(generator=gen).mul_(0.05)
    cache.s_bnd.normal_(generator=gen).mul_(0.05)
    cache.tail_k.normal_(generator=gen).mul_(0.09)
    cache.tail_v.normal_(generator=gen)
    cache.tail_g.uniform_(-1.0, -0.05, generator=gen)
    cache.tail_beta.uniform_(0.2, 0.8, generator=gen)
    cache.pos.copy_(torch.tensor(positions, dtype=torch.int32))
    return cache


def test_noalloc_decode_matches_workspace_decode(gdn):
    hqk, hv, d, C = 16, 32, 128, 64
    slots = 3
    # slot 0 completes its chunk on the first call, slot 1 on the second, slot 2 on neither
    positions = [C - 1, 2 * C - 2, 5]
    ref = make_cache(gdn, slots, hqk, hv, d, C, positions, seed=5)
    mine = make_cache(gdn, slots, hqk, hv, d, C, positions, seed=5)
    slot = torch.tensor([2, 0, 1], dtype=torch.int32, device="cuda")
    for call in range(2):
        x = synth.make_inputs([slots], hqk, hv, d, dtype=synth.BF16, seed=40 + call)
        t = {n: x[n].cuda() for n in ("q", "k", "v", "g", "beta")}
        o_ref = gdn.decode_step(t["q"], t["k"], t["v"], t["g"], t["beta"], slot, ref,
                                out_dtype=torch.float32)
        o = gdn.decode_step_noalloc(t["q"], t["k"], t["v"], t["g"], t["beta"], slot, mine,
                                    out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert rel_err(o, o_ref.double().cpu().numpy()) <= 2e-3
        assert torch.equal(o, o_ref), call
        for name in gdn.Cache.TENSORS:
            assert torch.equal(getattr(mine, name), getattr(ref, name)), (call, name)
    # slot 1 completed a chunk on the second call: its running state is the new boundary state
    assert torch.equal(mine.s_run[1], mine.s_bnd[1])
    assert mine.pos.tolist() == [C + 1, 2 * C, 7]


def test_noalloc_refuses_requests_beyond_its_scratch(gdn):
    lib = gdn.load()
    # 64 slots x 32 heads of d = 128, C = 64 needs about 128 MiB of decode workspace
    shape = gdn.make_shape(64, 64, 16, 32, 128, 64, torch.bfloat16, torch.bfloat16)
    need = gdn.workspace_bytes(shape, gdn.MODE_DECODE)
    assert need > gdn.NOALLOC_SCRATCH_BYTES
    fake = 1 << 20  # never dereferenced: the size check comes first and nothing is queued
    cache = gdn.CacheStruct(fake, fake, fake, fake, fake, fake, fake, fake, 64)
    rc = lib.gdn_cpr_decode_step_noalloc(ctypes.byref(shape), fake, fake, fake, fake, fake, fake,
                                         ctypes.byref(cache), fake, None)
    assert rc == 4  # GDN_ERR_WORKSPACE


def test_noalloc_device_errors_are_readable(gdn):
    """A slot index outside the cache is a device-side error; the no-alloc call records it in
    its built-in array's error word, which gdn_cpr_noalloc_device_error reads back.  The next
    valid call clears it."""
    hqk, hv, d, C = 2, 4, 64, 16
    cache = make_cache(gdn, 2, hqk, hv, d, C, [3, 20], seed=7)
    x = synth.make_inputs([2], hqk, hv, d, dtype=synth.BF16, seed=8)
    t = {n: x[n].cuda() for n in ("q", "k", "v", "g", "beta")}
    before = {n: getattr(cache, n).clone() for n in gdn.Cache.TENSORS}
    bad = torch.tensor([0, 5], dtype=torch.int32, device="cuda")
    gdn.decode_step_noalloc(t["q"], t["k"], t["v"], t["g"], t["beta"], bad, cache)
    assert gdn.noalloc_device_error() == 2  # GDN_DEVERR_SLOT
    # the valid slot 0 still stepped; slot 1 was not touched
    assert cache.pos.tolist() == [4, 20]
    for name in ("s_run", "s_bnd", "tail_g"):
        assert torch.equal(getattr(cache, name)[1], before[name][1]), name
    good = torch.tensor([1, 0], dtype=torch.int32, device="cuda")
    gdn.decode_step_noalloc(t["q"], t["k"], t["v"], t["g"], t["beta"], good, cache)
    assert gdn.noalloc_device_error() == 0
    assert cache.pos.tolist() == [5, 21]
