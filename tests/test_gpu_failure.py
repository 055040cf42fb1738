"""Failure paths that the device detects, exercised without a GPU fault.

- A bounded on-device wait that runs out: the test hook gdn_cpr_test_wait_timeout makes one
  CTA of the tensor-core boundary chain wait, before it issues any copy or MMA, on a barrier
  phase that nothing completes.  The wait gives up after a short poll limit, the CTA records
  GDN_DEVERR_TIMEOUT, frees its tensor memory and exits; gdn_cpr_get_device_error reports the
  code, and the next call on the same context runs normally and gives the usual bits.  (The
  hegai.media page, section "Что именно объединяет IsoExec": a configuration that cannot be
  verified is rejected rather than run; here a kernel that cannot finish reports so.)
- gdn_cpr_running_state with a slot index outside the cache gives an all-NaN block.
"""
import pytest
import torch

from gated_deltanet_cpr_gb300 import synth
from helpers import to_dev

pytestmark = pytest.mark.gpu


def prefill(gdn, t, x, ws):
    return gdn.prefill(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], chunk=64,
                       out_dtype=torch.float32, cu_seqlens_host=x["cu_seqlens"], ws=ws)


def test_bounded_wait_timeout_is_reported(gdn):
    lengths = [300, 64, 130]
    x = synth.make_inputs(lengths, 2, 4, 128, dtype=synth.BF16, seed=31, decay="slow")
    t = to_dev(x)
    shape = gdn.make_shape(3, sum(lengths), 2, 4, 128, 64, torch.bfloat16, torch.float32)
    ws = gdn.alloc_workspace(gdn.workspace_bytes(shape, gdn.MODE_PREFILL, x["cu_seqlens"]), "cuda")
    o_ref, st_ref = prefill(gdn, t, x, ws)
    o_ref, st_ref = o_ref.clone(), st_ref.clone()
    assert gdn.device_error(ws) == 0
    gdn.test_wait_timeout(1)
    try:
        prefill(gdn, t, x, ws)
        assert gdn.device_error(ws) == 4  # GDN_DEVERR_TIMEOUT
    finally:
        gdn.test_wait_timeout(0)
    o, st = prefill(gdn, t, x, ws)
    assert gdn.device_error(ws) == 0
    assert torch.equal(o, o_ref)
    assert torch.equal(st, st_ref)


def test_running_state_rejects_bad_slots_with_nan(gdn):
    cache = gdn.Cache(3, 2, 4, 32, 16, dtype=torch.bfloat16)
    cache.s_run.normal_()
    cache.c_run.fill_(0.5)
    out = cache.running_state(torch.tensor([2, 7, -1], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(out[0], cache.s_run[2] * 0.5)
    assert torch.isnan(out[1]).all() and torch.isnan(out[2]).all()
