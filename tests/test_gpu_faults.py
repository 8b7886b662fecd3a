"""Failure detection on the GPU without faulting it.

Every device-side wait is bounded.  The test hook AGMM_TEST_DROP_ARRIVE makes
the producer skip its first arrival, so the MMA thread's wait on that stage
runs out (here after 200 ms): the kernel records AGMM_ERR_TIMEOUT in the
workspace status words, every role leaves its loop, in-flight copies are
drained, tensor memory is freed and the kernel returns.  The host reads the
status through agmm_query_status, and the context stays usable: the next
normal run is correct.  Nothing here traps, asserts on the device or touches
an invalid address.
"""
import numpy as np
import pytest
import torch

import oracle
from all_gather_gemm_agmm_gb300.inputs import make_inputs

from parity import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def agmm():
    import all_gather_gemm_agmm_gb300 as m
    from all_gather_gemm_agmm_gb300 import _build

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _build.build()
    m.load_library()
    return m


@pytest.mark.parametrize("case", [(2, 16, 256, 128, False, "2"),     # swapped tiles, cluster split-K
                                  (3, 200, 512, 384, True, "2"),     # row tiles, clusters of two, stream-K
                                  (1, 300, 256, 256, False, "1")],   # row tiles, one CTA per cluster
                         ids=["swap", "rows_cluster", "rows_single"])
def test_dropped_arrival_times_out_and_recovers(agmm, case, monkeypatch):
    P, m, k, n, rt, cm = case
    monkeypatch.setenv("AGMM_CM", cm)
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=9)
    xs = [x.cuda() for x in xs_cpu]
    y = y_cpu.cuda()
    o = torch.zeros((P * m, n), dtype=torch.bfloat16, device="cuda")

    monkeypatch.setenv("AGMM_TEST_DROP_ARRIVE", "1")
    monkeypatch.setenv("AGMM_WAIT_LIMIT_MS", "200")
    bad = agmm.Plan(P, m, k, n, rt)
    monkeypatch.delenv("AGMM_TEST_DROP_ARRIVE")
    monkeypatch.delenv("AGMM_WAIT_LIMIT_MS")
    ws = bad.new_workspace()
    bad.run(xs, y, o, 0, ws)
    with pytest.raises(agmm.AgmmError) as err:
        bad.query_status(ws)
    assert err.value.status == agmm.AGMM_ERR_TIMEOUT
    assert "ran out" in str(err.value)
    # the status words were cleared by the query
    assert bad.query_status(ws) == agmm.AGMM_OK

    good = agmm.Plan(P, m, k, n, rt)
    ws2 = good.new_workspace()
    good.run(xs, y, o, 0, ws2)
    assert good.query_status(ws2) == agmm.AGMM_OK
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, rt)
    check(o, ref32, f"after a timeout {good.info()}")
