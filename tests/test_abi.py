"""The C ABI library builds for sm_103a, loads, and exports every entry
point that include/specv.h declares; host-side argument checks need no GPU."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_57_gb300 import _lib, build

    build.build()
    return _lib.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "specv.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(specv_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("specv_create", "specv_verify_sample", "specv_verify_greedy", "specv_destroy",
              "specv_status_string", "specv_verify_sample_host"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from speculative_decoding_verification_57_gb300 import build

    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(specv_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib, n)


def test_status_strings(lib):
    assert lib.specv_status_string(0) == b"ok"
    assert lib.specv_status_string(1) == b"invalid argument"
    assert lib.specv_status_string(99) == b"unknown status"


def test_argument_errors_need_no_device(lib):
    # a null handle is rejected before any CUDA call
    st = lib.specv_verify_sample(None, 1, None, None, None, None, None, 1, 4, 100, None, None, None, None, None)
    assert st == 1
    st = lib.specv_verify_greedy(None, 0, None, None, 1, 4, 100, None, None, None, None)
    assert st == 1
    assert lib.specv_plan_cluster(None, 1, 1, 4, 100) == 0
    assert lib.specv_launch_count(None) == 0
    lib.specv_destroy(None)
    h = ctypes.c_void_p()
    assert lib.specv_create(None, 0, 1, 4, 100) == 1
    assert lib.specv_create(ctypes.byref(h), 0, 1, 0, 100) == 1  # k < 1
    assert lib.specv_create(ctypes.byref(h), 0, 1, 32, 100) == 1  # k above 31
    assert lib.specv_create(ctypes.byref(h), 0, 1, 4, 0) == 1  # empty vocabulary
    assert lib.specv_create(ctypes.byref(h), 0, 1, 4, 262145) == 1  # vocabulary above 16 x 16384
    assert lib.specv_create(ctypes.byref(h), 0, -1, 4, 100) == 1  # negative batch


def test_kernels_are_built_for_sm_103a():
    from speculative_decoding_verification_57_gb300 import build

    assert build.ARCH == "-gencode=arch=compute_103a,code=sm_103a"
