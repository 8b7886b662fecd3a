"""The allocation-free entry point agmm_run_unfused_noalloc.

It serves callers that cannot allocate device memory where they run the
all-gather matmul: code under a framework allocator that has reserved the
device's memory for itself, and loops that cannot afford the implicit device
synchronisation of cudaMalloc and cudaFree.  Its scratch is a static device
array inside the library.  These tests call it through the C ABI, twice in a
row on the same static scratch, and compare its output with agmm_run_unfused
on a caller workspace and with the CPU oracle.  This file is collected last
so that a run stopping at the first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from all_gather_gemm_agmm_gb300.inputs import make_inputs

from parity import check

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 64 << 20  # AGMM_STATIC_SCRATCH_BYTES in include/agmm.h


@pytest.fixture(scope="module")
def agmm():
    import all_gather_gemm_agmm_gb300 as m
    from all_gather_gemm_agmm_gb300 import _build

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    m.load_library()
    return m


def _ptrs(ts):
    return (ctypes.c_void_p * len(ts))(*[ctypes.c_void_p(t.data_ptr()) for t in ts])


@pytest.mark.parametrize("case", [(4, 64, 4096, 1024, True), (3, 200, 512, 384, False), (8, 130, 1024, 640, True)],
                         ids=["swapped", "rows", "rows_tail"])
def test_noalloc_matches_unfused_twice(agmm, case):
    P, m, k, n, rt = case
    lib = agmm.load_library()
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=7)
    xs = [x.cuda() for x in xs_cpu]
    y = y_cpu.cuda()
    plan = agmm.Plan(P, m, k, n, rt)
    assert plan.workspace_bytes(unfused=True) <= STATIC_SCRATCH_BYTES
    stream = torch.cuda.current_stream()
    o_ref = torch.empty((P * m, n), dtype=torch.bfloat16, device="cuda")
    plan.run_unfused(xs, y, o_ref, P - 1, plan.new_workspace(True))
    torch.cuda.synchronize()
    ref = o_ref.float().cpu().numpy()
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, rt)
    for call in range(2):
        o = torch.full((P * m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = lib.agmm_run_unfused_noalloc(plan._h, _ptrs(xs), y.data_ptr(), o.data_ptr(), P - 1,
                                          stream.cuda_stream)
        assert rc == agmm.AGMM_OK, lib.agmm_last_error().decode()
        torch.cuda.synchronize()
        check(o, ref, f"no-alloc call {call} vs agmm_run_unfused")
        check(o, ref32, f"no-alloc call {call} vs the oracle")


def test_noalloc_rejects_oversized_problem(agmm):
    lib = agmm.load_library()
    plan = agmm.Plan(8, 1024, 8192, 1024, False)  # gathered X alone is 128 MiB
    assert plan.workspace_bytes(unfused=True) > STATIC_SCRATCH_BYTES
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    rc = lib.agmm_run_unfused_noalloc(plan._h, _ptrs([dummy] * 8), dummy.data_ptr(), dummy.data_ptr(), 0,
                                      torch.cuda.current_stream().cuda_stream)
    assert rc == agmm.AGMM_ERR_INVALID_ARG
    assert "static scratch" in lib.agmm_last_error().decode()
