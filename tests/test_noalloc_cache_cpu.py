"""Host logic of the no-alloc decode entry point's scratch-address cache, on the CPU.

The built-in scratch array's device address is cached per device together with the
identity of the context it was looked up in, so that after a device reset (a new context,
in which the array may sit elsewhere) the address is looked up again instead of reused.
This compiles a small C++ program around the cache with fake context identities and fake
lookups (no GPU, no CUDA) and checks each case.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_scratch_address_cache_logic(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = str(tmp_path / "noalloc_cache_test")
    src = os.path.join(HERE, "cpp", "noalloc_cache_test.cpp")
    subprocess.check_call([cxx, "-std=c++17", "-O1", "-pthread", "-o", exe, src])
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip() == "ok"
