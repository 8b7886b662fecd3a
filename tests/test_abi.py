"""The C ABI on the host: the library loads, exports every declared symbol,
and rejects bad shapes and arguments before touching a device."""
import ctypes
import os
import re

import pytest

import all_gather_gemm_agmm_gb300 as agmm

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "agmm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(agmm_[a-z_]+)\s*\(", text)))


def test_header_matches_binding_list():
    assert declared_functions() == sorted(agmm.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(agmm_lib):
    for name in declared_functions():
        assert hasattr(agmm_lib, name), name


def test_version_and_status_strings(agmm_lib):
    assert agmm_lib.agmm_version() == 1
    for code in range(7):
        assert agmm_lib.agmm_status_string(code).decode().startswith("AGMM_")
    assert agmm_lib.agmm_status_string(99).decode() == "AGMM_ERR_UNKNOWN"


def _plan(lib, P, m, k, n, dtype=0, rt=0):
    h = ctypes.c_void_p(12345)
    st = lib.agmm_plan(P, m, k, n, dtype, rt, ctypes.byref(h))
    return st, h


@pytest.mark.parametrize("args,why", [
    ((0, 16, 256, 128), "P < 1"),
    ((9, 16, 256, 128), "P > 8"),
    ((2, 0, 256, 128), "empty shard"),
    ((2, -1, 256, 128), "negative rows"),
    ((2, 16, 0, 128), "k = 0"),
    ((2, 16, 192, 128), "k % 128"),
    ((2, 16, 256, 64), "n < 128"),
    ((2, 16, 256, 200), "n % 128"),
    ((8, 1 << 31, 256, 128), "m >= 2^31"),
    ((8, 1 << 30, 1 << 20, 128), "operand above 2^40 elements"),
])
def test_plan_rejects_bad_shapes_before_cuda(agmm_lib, args, why):
    st, h = _plan(agmm_lib, *args)
    assert st == agmm.AGMM_ERR_INVALID_ARG, why
    assert h.value is None
    assert agmm_lib.agmm_last_error().decode()


def test_plan_rejects_bad_dtype_and_flag(agmm_lib):
    assert _plan(agmm_lib, 2, 16, 256, 128, dtype=7)[0] == agmm.AGMM_ERR_INVALID_ARG
    assert _plan(agmm_lib, 2, 16, 256, 128, dtype=-1)[0] == agmm.AGMM_ERR_INVALID_ARG
    assert _plan(agmm_lib, 2, 16, 256, 128, rt=2)[0] == agmm.AGMM_ERR_INVALID_ARG
    assert agmm_lib.agmm_plan(2, 16, 256, 128, 0, 0, None) == agmm.AGMM_ERR_INVALID_ARG


def test_null_plan_calls(agmm_lib):
    agmm_lib.agmm_destroy(None)  # no-op
    assert agmm_lib.agmm_workspace_bytes(None, 0) == 0
    arr = (ctypes.c_void_p * 1)()
    assert agmm_lib.agmm_run(None, arr, None, None, 0, None, None) == agmm.AGMM_ERR_INVALID_ARG
    assert agmm_lib.agmm_run_unfused(None, arr, None, None, 0, None, None) == agmm.AGMM_ERR_INVALID_ARG
    assert agmm_lib.agmm_run_gather(None, arr, None, None, None, 0, None, None) == agmm.AGMM_ERR_INVALID_ARG
    assert agmm_lib.agmm_plan_info(None, None) == agmm.AGMM_ERR_INVALID_ARG
    assert agmm_lib.agmm_query_status(None, None, None) == agmm.AGMM_ERR_INVALID_ARG


def test_valid_shape_without_device_is_a_cuda_error(agmm_lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a device is present")
    st, h = _plan(agmm_lib, 2, 16, 256, 128)
    assert st == agmm.AGMM_ERR_CUDA and h.value is None


def test_ring_chunks_argument_checks(agmm_lib):
    n = ctypes.c_int64(0)
    f = agmm_lib.agmm_ring_chunks
    assert f(0, 4, 0, 8, 0, None, None, None, None, 0, ctypes.byref(n)) == agmm.AGMM_ERR_INVALID_ARG
    assert f(2, 4, 2, 8, 0, None, None, None, None, 0, ctypes.byref(n)) == agmm.AGMM_ERR_INVALID_ARG
    assert f(2, 0, 0, 8, 0, None, None, None, None, 0, ctypes.byref(n)) == agmm.AGMM_ERR_INVALID_ARG
    assert f(2, 4, 0, 0, 0, None, None, None, None, 0, ctypes.byref(n)) == agmm.AGMM_ERR_INVALID_ARG
    assert f(2, 4, 0, 8, 2, None, None, None, None, 0, ctypes.byref(n)) == agmm.AGMM_ERR_INVALID_ARG
    assert f(2, 4, 0, 8, 0, None, None, None, None, 0, None) == agmm.AGMM_ERR_INVALID_ARG
    assert f(2, 4, 0, 8, 0, None, None, None, None, 0, ctypes.byref(n)) == agmm.AGMM_OK
    assert n.value == 2 * 2
    assert f(2, 4, 0, 8, 1, None, None, None, None, 0, ctypes.byref(n)) == agmm.AGMM_OK
    assert n.value == 2


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(ImportError):
        agmm.load_library(str(tmp_path / "libagmm.so"))
