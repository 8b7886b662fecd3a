"""GPU tests of the tuner (tune.py) and of the 2-D Y loads that the 3-D
tensor map replaces for Y stored [k, n] (kept for drivers that refuse the 3-D
map, and selected here with AGMM_Y3D=0)."""
import pytest
import torch

import oracle
from all_gather_gemm_agmm_gb300.inputs import WORKLOADS, make_inputs

from parity import alloc_output_guarded, check, guards_intact, to_device_guarded

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


def test_tune_shape_end_to_end(agmm):
    # the tiny workload with short timings: every candidate plans, matches the
    # planner's choice on NaN-poisoned output and is timed
    from all_gather_gemm_agmm_gb300 import tune

    rec = tune.tune_shape(WORKLOADS["c1_tiny"], screen_s=0.005, final_s=0.01, rounds=1)
    assert rec["name"] == "c1_tiny" and rec["rules"]["us"] > 0 and rec["best"]["us"] > 0
    timed = [t for t in rec["trials"] if "screen_us" in t]
    assert len(timed) >= 4
    assert not [t for t in rec["trials"] if "error" in t], rec["trials"]
    assert rec["best"]["us"] <= rec["rules"]["us"]
    if rec["tuned"]:
        assert rec["best"]["us"] <= rec["rules"]["us"] * (1 - tune.MARGIN)


@pytest.mark.parametrize("case", [(3, 200, 512, 768), (4, 64, 1024, 512), (8, 8, 512, 256)],
                         ids=lambda c: "P{}_m{}_k{}_n{}".format(*c))
def test_two_d_y_loads_match_oracle(agmm, case, monkeypatch):
    # Y stored [k, n] through one 2-D box per 64 columns (row and swapped tiles)
    monkeypatch.setenv("AGMM_Y3D", "0")
    P, m, k, n = case
    xs_cpu, y_cpu = make_inputs(P, m, k, n, False, seed=41)
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, False)
    xs = [to_device_guarded(x)[0] for x in xs_cpu]
    y, _ = to_device_guarded(y_cpu)
    o, obuf = alloc_output_guarded(P * m, n)
    plan = agmm.Plan(P, m, k, n, False)
    ws = plan.new_workspace()
    torch.cuda.synchronize()
    plan.run(xs, y, o, P - 1, ws)
    plan.query_status(ws)
    torch.cuda.synchronize()
    assert guards_intact(obuf)
    check(o, ref32, f"2-D Y loads {case} {plan.info()}")
