"""CPU-only checks of the C-ABI library: it loads, exports every function the header
declares, and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest
import torch

from gated_deltanet_cpr_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn_cpr.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:gdn_status|int|void|const char\s*\*)\s*(gdn_cpr_\w+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_abi():
    names = declared_functions()
    assert set(api.EXPORTS) <= set(names), names
    assert len(names) >= 8


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.gdn_cpr_version() >= 100
    assert lib.gdn_cpr_status_string(2) == b"unsupported configuration"


def shape(**kw):
    base = dict(num_seqs=2, total_tokens=100, h_qk=2, h_v=4, d=64, chunk=32,
                in_dtype=torch.bfloat16, out_dtype=torch.bfloat16)
    base.update(kw)
    return api.make_shape(base["num_seqs"], base["total_tokens"], base["h_qk"], base["h_v"],
                          base["d"], base["chunk"], base["in_dtype"], base["out_dtype"])


def ws_size(lib, sh, mode, cu):
    n = ctypes.c_size_t(0)
    cu_t = None if cu is None else torch.tensor(cu, dtype=torch.int32)
    rc = lib.gdn_cpr_workspace_size(ctypes.byref(sh), mode, None if cu_t is None else cu_t.data_ptr(),
                                    ctypes.byref(n))
    return rc, n.value


def test_workspace_size_and_claims(lib):
    rc, n = ws_size(lib, shape(), api.MODE_PREFILL, [0, 60, 100])
    assert rc == 0 and n > 0 and n % 256 == 0
    rc2, n2 = ws_size(lib, shape(), api.MODE_FWD, [0, 60, 100])
    assert rc2 == 0 and n2 < n  # the trainer forward keeps boundary states in saved_bnd
    rc, n = ws_size(lib, shape(num_seqs=8, total_tokens=8), api.MODE_DECODE, None)
    assert rc == 0 and n > 0
    # unsupported configurations (claims)
    assert ws_size(lib, shape(d=96), api.MODE_PREFILL, [0, 60, 100])[0] == 2
    assert ws_size(lib, shape(chunk=48), api.MODE_PREFILL, [0, 60, 100])[0] == 2
    assert ws_size(lib, shape(h_qk=3, h_v=4), api.MODE_PREFILL, [0, 60, 100])[0] == 2
    # bad cu_seqlens on the host
    assert ws_size(lib, shape(), api.MODE_PREFILL, [0, 60, 99])[0] == 1
    assert ws_size(lib, shape(), api.MODE_PREFILL, [1, 60, 100])[0] == 1
    assert ws_size(lib, shape(), api.MODE_PREFILL, [0, 70, 60])[0] == 1
    assert ws_size(lib, shape(), api.MODE_PREFILL, None)[0] == 1


def test_prefill_rejects_bad_arguments_before_any_launch(lib):
    sh = shape()
    cu = torch.tensor([0, 60, 100], dtype=torch.int32)
    fake = 1 << 20  # 16-byte aligned, never dereferenced: checks fail first
    args = dict(q=fake, k=fake, v=fake, g=fake, beta=fake, state_in=None, cu_dev=fake,
                cu_host=cu.data_ptr(), o=fake, state_out=None, cache=None, slot=None, ws=fake,
                ws_bytes=0, stream=None)

    def call(**over):
        a = dict(args)
        a.update(over)
        return lib.gdn_cpr_prefill(ctypes.byref(a.pop("shape", sh)), a["q"], a["k"], a["v"],
                                   a["g"], a["beta"], a["state_in"], a["cu_dev"], a["cu_host"],
                                   a["o"], a["state_out"], a["cache"], a["slot"], a["ws"],
                                   a["ws_bytes"], a["stream"])

    assert call() == 4                      # workspace too small
    assert call(q=None) == 1                # null input
    assert call(k=fake + 2) == 1            # misaligned input
    assert call(shape=shape(d=48)) == 2     # unsupported head dim
    assert call(ws=fake + 16, ws_bytes=1 << 40) == 4  # misaligned workspace
    bad = torch.tensor([0, 60, 90], dtype=torch.int32)
    assert call(cu_host=bad.data_ptr()) == 1


def test_decode_and_bwd_argument_checks(lib):
    sh = shape(num_seqs=4, total_tokens=5)
    cache = api.CacheStruct(1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 4)
    fake = 1 << 20
    rc = lib.gdn_cpr_decode_step(ctypes.byref(sh), fake, fake, fake, fake, fake, fake,
                                 ctypes.byref(cache), fake, fake, 1 << 30, None)
    assert rc == 1  # total_tokens must equal num_seqs for a decode step
    sh = shape(num_seqs=4, total_tokens=4)
    cache.slots = 0
    rc = lib.gdn_cpr_decode_step(ctypes.byref(sh), fake, fake, fake, fake, fake, fake,
                                 ctypes.byref(cache), fake, fake, 1 << 30, None)
    assert rc == 1  # empty cache
    rc = lib.gdn_cpr_get_device_error(None, None, None)
    assert rc == 1


def test_checked_build_exports_every_declared_symbol():
    """The bounds-checked debug variant (GDN_CHECKED=1) builds and exports the same ABI."""
    import ctypes as ct

    path = build.build(checked=True)
    assert path.endswith("libgdn_cpr_checked.so")
    lib = ct.CDLL(path)
    for name in declared_functions():
        assert hasattr(lib, name), name
