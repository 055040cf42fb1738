"""GPU parity of the CPR forward (prefill / trainer forward) against the fp64 oracle.

Tolerances: max|GPU - oracle| / max|oracle| per output tensor, <= 1e-5 for fp32 inputs and
<= 2e-3 for bf16 inputs.  The oracle is the token-by-token recurrence of the gated delta
rule (IsoExec page, section "Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet"); the CPR
path evaluates it with a chunked boundary pass plus per-chunk recurrences, so only
rounding differs.
"""
import numpy as np
import pytest
import torch

from gated_deltanet_cpr_gb300 import synth
from helpers import oracle_full, oracle_pairs, rel_err, to_dev

pytestmark = pytest.mark.gpu

TOL = {synth.F32: 1e-5, synth.BF16: 2e-3}
TD = {synth.F32: torch.float32, synth.BF16: torch.bfloat16}


def run_prefill(gdn, x, C, out=torch.float32):
    t = to_dev(x)
    return gdn.prefill(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], chunk=C,
                       state_in=t["state_in"], out_dtype=out, cu_seqlens_host=x["cu_seqlens"])


def test_tiny_fp32_full_oracle(gdn):
    """B=1, H=2, T=256, d=32, C=16, fp32: every output against the oracle."""
    w = synth.workloads()["tiny"]
    x = synth.make_inputs(w.lengths, w.h_qk, w.h_v, w.d, dtype=w.dtype, seed=0)
    o, st = run_prefill(gdn, x, w.chunk)
    o_ref, st_ref, _ = oracle_full(x)
    assert rel_err(o, o_ref) <= TOL[synth.F32]
    assert rel_err(st, st_ref) <= TOL[synth.F32]


@pytest.mark.parametrize("d,C", [(32, 16), (64, 32), (128, 64), (128, 16), (64, 64)])
@pytest.mark.parametrize("dtype", [synth.BF16, synth.F32])
def test_ragged_batches(gdn, d, C, dtype):
    """Ragged lengths spanning several chunks, a tail, single tokens and empty sequences."""
    lengths = [1, C - 1, C, C + 1, 3 * C + 5, 0, 2 * C]
    x = synth.make_inputs(lengths, 2, 4, d, dtype=dtype, seed=d + C, state_in=True)
    o, st = run_prefill(gdn, x, C)
    o_ref, st_ref, _ = oracle_full(x)
    assert rel_err(o, o_ref) <= TOL[dtype], rel_err(o, o_ref)
    assert rel_err(st, st_ref) <= TOL[dtype], rel_err(st, st_ref)
    # empty sequence: state passes through bit for bit
    assert torch.equal(st[5], x["state_in"][5].cuda())


@pytest.mark.parametrize("dtype", [synth.BF16, synth.F32])
def test_slow_decay_carries_memory(gdn, dtype):
    """g = -0.02 sigmoid(N(0,1)): boundary states carry memory across many chunks."""
    lengths = [700, 333, 64]
    x = synth.make_inputs(lengths, 2, 4, 64, dtype=dtype, seed=3, decay="slow", state_in=True)
    o, st = run_prefill(gdn, x, 64)
    o_ref, st_ref, _ = oracle_full(x)
    assert rel_err(o, o_ref) <= TOL[dtype], rel_err(o, o_ref)
    assert rel_err(st, st_ref) <= TOL[dtype], rel_err(st, st_ref)


def test_boundary_states_match_oracle(gdn):
    """The trainer forward's saved boundary states S^(j) against the recurrence's state
    before every chunk."""
    lengths = [130, 64, 7, 0, 200]
    x = synth.make_inputs(lengths, 2, 4, 64, dtype=synth.BF16, seed=4, decay="slow", state_in=True)
    t = to_dev(x)
    o, st, bnd = gdn.fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], chunk=32,
                         state_in=t["state_in"], out_dtype=torch.float32,
                         cu_seqlens_host=x["cu_seqlens"])
    _, _, bnd_ref = oracle_full(x, chunk=32)
    assert bnd.shape[0] == bnd_ref.shape[0]
    assert rel_err(bnd, bnd_ref) <= 2e-3


def test_bf16_output_is_rounded_fp32_output(gdn):
    lengths = [100, 37]
    x = synth.make_inputs(lengths, 2, 4, 64, dtype=synth.BF16, seed=5)
    o32, _ = run_prefill(gdn, x, 32, out=torch.float32)
    o16, _ = run_prefill(gdn, x, 32, out=torch.bfloat16)
    assert torch.equal(o16, o32.to(torch.bfloat16))


def test_chunk_size_independence(gdn):
    """Different C give the same function up to rounding."""
    lengths = [300, 129]
    x = synth.make_inputs(lengths, 2, 4, 64, dtype=synth.F32, seed=6, decay="slow")
    outs = [run_prefill(gdn, x, C)[0] for C in (16, 32, 64)]
    for o in outs[1:]:
        assert rel_err(o, outs[0].double().cpu().numpy()) <= 1e-5


def test_full_size_prefill_sampled_pairs(gdn):
    """The full prefill workload (4 x 4096 tokens, 16/32 heads, d=128, C=64, bf16) in the
    launch configuration the benchmark times, checked on a seeded sample of
    (sequence, head) pairs that the oracle recomputes one by one."""
    w = synth.workloads()["prefill"]
    x = synth.make_inputs(w.lengths, w.h_qk, w.h_v, w.d, dtype=w.dtype, seed=0)
    o, st = run_prefill(gdn, x, w.chunk, out=torch.bfloat16)
    o32, _ = run_prefill(gdn, x, w.chunk, out=torch.float32)
    assert torch.equal(o, o32.to(torch.bfloat16))
    rng = np.random.default_rng(0)
    pairs = [(int(rng.integers(4)), int(rng.integers(32))) for _ in range(8)]
    ref = oracle_pairs(x, pairs)
    cu = x["cu_seqlens"].tolist()
    for (s, h), (o_ref, st_ref, _) in ref.items():
        assert rel_err(o32[cu[s]:cu[s + 1], h], o_ref) <= 2e-3, (s, h)
        assert rel_err(st[s, h], st_ref) <= 2e-3, (s, h)
    assert torch.isfinite(o32).all()
