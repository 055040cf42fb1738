"""gdn_cpr_policy_digest (numerical-policy identity, IsoExec pages, section on the structure
of the execution contract, item "Identities"), on the CPU.

- The digest is SHA-256 of the returned canonical text, checked against Python's hashlib
  (an independent implementation; the ~1 KB text spans many 64-byte blocks).
- Everything that leaves the bits unchanged is outside the digest: number of sequences,
  tokens, heads and the head grouping.
- Everything that changes the bits changes the digest: head dimension, chunk length,
  input and output dtypes, and with them the boundary path (tensor cores only for bf16
  inputs at d = 128, C = 64).
- Shapes the calls reject are rejected here with the same status.
"""
import hashlib
import itertools

import pytest
import torch

from gated_deltanet_cpr_gb300 import api

BF, F32 = torch.bfloat16, torch.float32
UNSUPPORTED = 2  # gdn_status GDN_ERR_UNSUPPORTED


@pytest.fixture(scope="module")
def lib():
    return api.load()


@pytest.mark.parametrize("d,C,dt", [(128, 64, BF), (128, 64, F32), (32, 16, F32), (64, 32, BF)])
def test_digest_is_sha256_of_the_text(lib, d, C, dt):
    h, text = api.policy_digest(d, C, dt)
    assert len(text) > 700
    assert h == hashlib.sha256(text.encode()).hexdigest()
    assert f"d_k={d}\n" in text and f"chunk={C}\n" in text


def test_digest_ignores_batch_and_heads(lib):
    ref = api.policy_digest(128, 64, BF)[0]
    for n, T, hqk, hv in [(1, 0, 1, 1), (4, 16384, 16, 32), (256, 256, 32, 32), (7, 999, 8, 64)]:
        assert api.policy_digest(128, 64, BF, h_qk=hqk, h_v=hv, num_seqs=n, total_tokens=T)[0] == ref


def test_digest_separates_policies(lib):
    seen = {}
    for d, C, din, dout in itertools.product((32, 64, 128), (16, 32, 64), (BF, F32), (BF, F32)):
        h, text = api.policy_digest(d, C, din, dout)
        assert h not in seen, (seen.get(h), (d, C, din, dout))
        seen[h] = (d, C, din, dout)
        assert ("tcgen05" in text) == (din == BF and d == 128 and C == 64)
    assert len(seen) == 36


def test_digest_rejects_what_the_calls_reject(lib):
    with pytest.raises(api.GdnError) as e:
        api.policy_digest(96, 64, BF)
    assert e.value.code == UNSUPPORTED
    with pytest.raises(api.GdnError) as e:
        api.policy_digest(128, 48, BF)
    assert e.value.code == UNSUPPORTED
    with pytest.raises(api.GdnError) as e:
        api.policy_digest(128, 64, BF, h_qk=3, h_v=4)
    assert e.value.code == UNSUPPORTED
