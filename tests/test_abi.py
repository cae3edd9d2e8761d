"""The C ABI without a GPU: the library builds and loads, exports every function
include/cfa.h declares, and rejects bad arguments on the host before touching
the device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cfa.h")


@pytest.fixture(scope="module")
def lib():
    from out_proj_block_gb300 import build
    build.build()
    from out_proj_block_gb300 import cfa
    return cfa


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(cfa_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("cfa_plan_create", "cfa_decode_step", "cfa_plan_destroy"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    dll = ctypes.CDLL(lib.LIB_PATH)
    for name in declared_functions():
        assert hasattr(dll, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (cfa_\w+)", out))
    assert set(declared_functions()) <= exported
    assert set(lib.EXPORTED_SYMBOLS) == set(declared_functions())


def test_status_strings(lib):
    assert lib.cfa_status_string(0) == "CFA_OK"
    assert lib.cfa_status_string(4) == "CFA_ERR_TIMEOUT"
    assert lib.cfa_status_string(99) == "CFA_ERR_UNKNOWN"


@pytest.mark.parametrize("args,code", [
    ((0, 4096, 32, 128, 64), 1),        # B < 1
    ((1, 4096, 32, 100, 64), 1),        # hidden != n_heads * head_dim
    ((1, 4096, 32, 128, 0), 1),         # max_ctx < 1
    ((17, 4096, 32, 128, 64), 2),       # B > 16
    ((1, 3200, 32, 100, 64), 2),        # head_dim not 64/128
    ((1, 96, 1, 96, 64), 2),            # head_dim 96
    ((1, 4096, 32, 128, (1 << 22) + 1), 2),
])
def test_plan_create_rejects_bad_shapes_on_host(lib, args, code):
    assert lib._lib.cfa_plan_create(*args) is None
    assert lib.cfa_last_error() == code


def test_null_plan_is_rejected(lib):
    assert lib._lib.cfa_decode_step(None, 16, 16, 16, 16, 16, 0, 16, None) == lib.CFA_ERR_INVALID_ARG
    assert lib._lib.cfa_decode_step_host(None, 16, 16, 16, 16, 16, 0, 16, None) == lib.CFA_ERR_INVALID_ARG
    assert lib._lib.cfa_decode_step_ex(None, 16, 16, 16, 16, 16, None, 0.0, 16, None) == lib.CFA_ERR_INVALID_ARG
    assert lib._lib.cfa_plan_set_cluster_size(None, 2) == lib.CFA_ERR_INVALID_ARG
    assert lib._lib.cfa_plan_set_stages(None, 2) == lib.CFA_ERR_INVALID_ARG
    assert lib._lib.cfa_plan_set_overlap(None, 1) == lib.CFA_ERR_INVALID_ARG
    assert lib._lib.cfa_plan_cluster_size(None) == -1
    assert lib._lib.cfa_plan_status(None) == lib.CFA_ERR_INVALID_ARG
    buf = ctypes.create_string_buffer(8)
    assert lib._lib.cfa_plan_describe(None, buf, 8) == lib.CFA_ERR_INVALID_ARG
    lib._lib.cfa_plan_destroy(None)  # no-op


def test_selftest_rejects_bad_limit(lib):
    assert lib._lib.cfa_selftest_wait_timeout(0, None) == lib.CFA_ERR_INVALID_ARG
    assert lib._lib.cfa_selftest_wait_timeout((1 << 20) + 1, None) == lib.CFA_ERR_INVALID_ARG


def test_valid_plan_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib._lib.cfa_plan_create(1, 256, 2, 128, 128) is None
    assert lib.cfa_last_error() == lib.CFA_ERR_CUDA
