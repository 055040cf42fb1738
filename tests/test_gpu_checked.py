"""The bounds-checked debug build (GDN_CHECKED=1; the sanitizer stand-in on this hardware).

Every kernel of that build checks the index ranges it derives from device data (chunk and
sequence records, slots, positions) against the buffers it was given and records
GDN_DEVERR_BOUNDS instead of touching memory outside them.  Prefill on the tensor-core and
SIMT boundary paths, trainer forward and backward, decode through two resynchronisations and
a continued prefill run through it in a child process (GDN_CPR_CHECKED=1 selects the
library); no call may record a device error, and every output must equal the ordinary
build's bit for bit (the checks skip nothing on valid input and change no arithmetic)."""
import os
import subprocess
import sys

import pytest
import torch

from gated_deltanet_cpr_gb300 import build

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_checked_build_runs_clean_and_bit_identical(gdn, tmp_path):
    build.build(checked=True)
    out = str(tmp_path / "checked.pt")
    env = dict(os.environ, GDN_CPR_CHECKED="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "checked_cases.py"), out], env=env, cwd=HERE,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    got = torch.load(out)
    assert got["lib"].endswith("libgdn_cpr_checked.so")
    bad = {k: v for k, v in got["errs"].items() if v != 0}
    assert not bad, bad
    import checked_cases

    ref, ref_errs = checked_cases.run_cases()
    assert all(v == 0 for v in ref_errs.values())
    assert set(ref) == set(got["res"])
    for k in ref:
        assert torch.equal(ref[k], got["res"][k]), k
