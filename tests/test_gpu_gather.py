"""GPU tests of agmm_run_gather: the fused path that also writes the gathered
left-hand side concat(X_0 .. X_{P-1}) (the by-product of page 1's note on
splitting n).  The gathered buffer must equal the concatenation bit for bit,
with nothing written outside it, and O must meet the same parity gate as
agmm_run."""
import numpy as np
import pytest
import torch

import oracle
from all_gather_gemm_agmm_gb300.inputs import make_inputs

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


def _run_gather(agmm, xs_cpu, y_cpu, rt, my_id, f16=False):
    P = len(xs_cpu)
    m, k = xs_cpu[0].shape
    n = y_cpu.shape[0] if rt else y_cpu.shape[1]
    xs = [to_device_guarded(x)[0] for x in xs_cpu]
    y, _ = to_device_guarded(y_cpu)
    o, obuf = alloc_output_guarded(P * m, n, f16=f16)
    xcat, xbuf = alloc_output_guarded(P * m, k, f16=f16)
    plan = agmm.Plan(P, m, k, n, rt, f16=f16)
    ws = plan.new_workspace()
    plan.run_gather(xs, y, o, xcat, my_id, ws)
    plan.query_status(ws)
    torch.cuda.synchronize()
    assert guards_intact(obuf), "a store landed outside O"
    assert guards_intact(xbuf), "a store landed outside the gathered buffer"
    return o, xcat, plan


CASES = [
    # P, m_pd, k, n, rt: swapped tiles (whole-shard chunks, ragged), row tiles
    # (half-shard chunks, ragged halves, stream-K, clusters of two), odd shards
    (2, 16, 256, 128, False),
    (4, 64, 4096, 1024, True),
    (8, 8, 1024, 256, False),
    (3, 13, 256, 256, True),
    (3, 200, 512, 384, False),
    (2, 300, 256, 512, True),
    (5, 77, 1024, 256, False),
    (8, 130, 256, 640, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "P{}_m{}_k{}_n{}_{}".format(*c[:4], "rt" if c[4] else "nt"))
def test_gathered_lhs_exact(agmm, case):
    P, m, k, n, rt = case
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=11)
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, rt)
    o, xcat, plan = _run_gather(agmm, xs_cpu, y_cpu, rt, my_id=P // 2)
    want = torch.cat(xs_cpu).view(torch.int16)
    assert torch.equal(xcat.cpu().view(torch.int16), want), plan.info()
    check(o, ref32, f"{case} with gathered LHS {plan.info()}")


@pytest.mark.parametrize("mode", ["half", "whole"])
def test_gathered_lhs_chunking_modes(agmm, mode, monkeypatch):
    monkeypatch.setenv("AGMM_CHUNKS", mode)
    for (P, m, k, n, rt) in [(3, 200, 512, 384, False), (8, 8, 512, 256, True)]:
        xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=12)
        o, xcat, plan = _run_gather(agmm, xs_cpu, y_cpu, rt, my_id=1)
        assert torch.equal(xcat.cpu().view(torch.int16), torch.cat(xs_cpu).view(torch.int16)), (mode, plan.info())


def test_gathered_lhs_f16(agmm):
    P, m, k, n, rt = 4, 64, 1024, 512, True
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=13, dtype="f16")
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, rt)
    o, xcat, _ = _run_gather(agmm, xs_cpu, y_cpu, rt, my_id=3, f16=True)
    assert torch.equal(xcat.cpu().view(torch.int16), torch.cat(xs_cpu).view(torch.int16))
    check(o, ref32, "f16 with gathered LHS")


def test_gathered_lhs_same_o_as_run(agmm):
    # storing the gathered rows does not change the product
    P, m, k, n, rt = 3, 200, 512, 384, False
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=14)
    o_g, _, plan = _run_gather(agmm, xs_cpu, y_cpu, rt, my_id=2)
    xs = [x.cuda() for x in xs_cpu]
    o = torch.empty_like(o_g)
    ws = plan.new_workspace()
    torch.cuda.synchronize()
    plan.run(xs, y_cpu.cuda(), o, 2, ws)
    plan.query_status(ws)
    assert torch.equal(o.view(torch.int16), o_g.view(torch.int16))


def test_all_gather_matmul_returns_gathered(agmm):
    xs_cpu, y_cpu = make_inputs(4, 32, 512, 256, False, seed=15)
    o, xcat = agmm.all_gather_matmul([x.cuda() for x in xs_cpu], y_cpu.cuda(), my_id=1, return_gathered=True)
    torch.cuda.synchronize()
    assert torch.equal(xcat.cpu().view(torch.int16), torch.cat(xs_cpu).view(torch.int16))
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, False)
    check(o, ref32, "all_gather_matmul return_gathered")


def test_gathered_lhs_argument_errors_and_pair_plans(agmm):
    P, m, k, n = 2, 16, 256, 128
    xs_cpu, y_cpu = make_inputs(P, m, k, n, False, seed=16)
    xs = [x.cuda() for x in xs_cpu]
    y = y_cpu.cuda()
    o = torch.empty((P * m, n), dtype=torch.bfloat16, device="cuda")
    plan = agmm.Plan(P, m, k, n, False)
    ws = plan.new_workspace()
    torch.cuda.synchronize()
    # the gathered buffer may not overlap a shard
    with pytest.raises(agmm.AgmmError) as err:
        plan.run_gather(xs, y, o, xs[0], 0, ws)
    assert err.value.status == agmm.AGMM_ERR_INVALID_ARG
    # a CTA-pair plan (the row-tile default): each CTA's epilogue warps copy
    # its own rows
    pm, pk, pn = 256, 512, 256
    xs2, y2 = make_inputs(2, pm, pk, pn, False, seed=17)
    pplan = agmm.Plan(2, pm, pk, pn, False, config={"path": "rows", "cluster_m": 2, "cta_pair": True})
    assert pplan.info()["cta_pair"] == 1
    o2 = torch.empty((2 * pm, pn), dtype=torch.bfloat16, device="cuda")
    xc = torch.empty((2 * pm, pk), dtype=torch.bfloat16, device="cuda")
    ws2 = pplan.new_workspace()
    torch.cuda.synchronize()
    pplan.run_gather([x.cuda() for x in xs2], y2.cuda(), o2, xc, 0, ws2)
    pplan.query_status(ws2)
    torch.cuda.synchronize()
    assert torch.equal(xc.cpu().view(torch.int16), torch.cat(xs2).view(torch.int16))
    ref32, _ = oracle.agmm(xs2, y2, False)
    check(o2, ref32, "CTA-pair plan with gathered LHS")


ROW_FORMS = [
    {"path": "rows"},                                   # CTA pairs (the default)
    {"path": "rows", "cluster_m": 1},                   # one CTA per cluster
    {"path": "rows", "stages": 2},                      # a short ring: refills wait on the stores
    {"path": "rows", "stream_k": True, "group_m": 3},   # k blocks of the last wave shared
]
ROW_SHAPES = [
    (4, 512, 1024, 4096, True),    # 16 row tiles x 16 n tiles: several tiles per cluster, 1 k block stored per tile
    (3, 200, 2048, 384, False),    # ragged halves, odd row-tile count (an idle pair follower)
    (5, 77, 768, 1280, True),      # odd shards, 5 n tiles of 256
]


@pytest.mark.parametrize("cfg", ROW_FORMS, ids=str)
@pytest.mark.parametrize("shape", ROW_SHAPES, ids=lambda c: "P{}_m{}_k{}_n{}".format(*c[:4]))
def test_gathered_lhs_row_tile_forms(agmm, cfg, shape):
    # Row tiles copy the gathered LHS from the shards with the epilogue warps
    # while the main loop runs; the gathered buffer is exact and O is bitwise
    # the plain run's O under the same plan.
    P, m, k, n, rt = shape
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=18)
    plan = agmm.Plan(P, m, k, n, rt, config=cfg)
    info = plan.info()
    assert info["path"] == 0
    xs = [to_device_guarded(x)[0] for x in xs_cpu]
    y, _ = to_device_guarded(y_cpu)
    o_g, obuf = alloc_output_guarded(P * m, n)
    xcat, xbuf = alloc_output_guarded(P * m, k)
    o = torch.empty_like(o_g)
    ws = plan.new_workspace()
    torch.cuda.synchronize()
    for _ in range(2):  # a second run on the same workspace
        plan.run_gather(xs, y, o_g, xcat, P - 1, ws)
        plan.query_status(ws)
    plan.run(xs, y, o, P - 1, ws)
    plan.query_status(ws)
    torch.cuda.synchronize()
    assert guards_intact(obuf) and guards_intact(xbuf), info
    assert torch.equal(xcat.cpu().view(torch.int16), torch.cat(xs_cpu).view(torch.int16)), info
    assert torch.equal(o.view(torch.int16), o_g.view(torch.int16)), info
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, rt)
    check(o_g, ref32, f"{shape} {cfg} {info}")
