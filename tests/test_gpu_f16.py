"""GPU parity of the fp16 variant: fp16 shards and Y (the AllGather-GEMM
tutorial's float16 tensors), float32 accumulation, fp16 or float32 output,
through the C ABI, against the oracle's fp16 definition."""
import numpy as np
import pytest
import torch

import oracle
from all_gather_gemm_agmm_gb300.inputs import WORKLOADS, make_inputs

from parity import alloc_output_guarded, check, check_blocks, guards_intact, oracle_rows, to_device_guarded

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


def _run(agmm, xs_cpu, y_cpu, rt, my_id, f32=False, unfused=False):
    P = len(xs_cpu)
    m, k = xs_cpu[0].shape
    n = y_cpu.shape[0] if rt else y_cpu.shape[1]
    xs = [to_device_guarded(x)[0] for x in xs_cpu]
    y, _ = to_device_guarded(y_cpu)
    o, obuf = alloc_output_guarded(P * m, n, f32, f16=True)
    plan = agmm.Plan(P, m, k, n, rt, f32, f16=True)
    ws = plan.new_workspace(unfused)
    (plan.run_unfused if unfused else plan.run)(xs, y, o, my_id, ws)
    plan.query_status(ws)
    torch.cuda.synchronize()
    assert guards_intact(obuf), "a store landed outside O"
    return o, plan


CASES = [
    # P, m_pd, k, n, rt, dist: swapped tiles, row tiles, ragged halves, both layouts
    (2, 16, 256, 128, False, "uniform"),
    (4, 64, 4096, 1024, True, "normal"),
    (8, 8, 1024, 256, False, "normal"),
    (3, 5, 128, 128, True, "normal"),
    (3, 200, 512, 384, False, "normal"),
    (2, 300, 256, 512, True, "normal"),
    (5, 77, 384, 256, False, "uniform"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "P{}_m{}_k{}_n{}_{}".format(*c[:4], "rt" if c[4] else "nt"))
def test_f16_parity(agmm, case):
    P, m, k, n, rt, dist = case
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, dist=dist, seed=0, dtype="f16")
    ref32, ref16 = oracle.agmm(xs_cpu, y_cpu, rt)
    o, plan = _run(agmm, xs_cpu, y_cpu, rt, my_id=P - 1)
    assert o.dtype == torch.float16
    check(o, ref32, f"{case} f16 {plan.info()}")
    # most elements round to exactly the oracle's fp16 value
    same = np.mean(o.cpu().view(torch.int16).numpy().view(np.uint16) == ref16)
    assert same > 0.9, same
    o32, _ = _run(agmm, xs_cpu, y_cpu, rt, my_id=0, f32=True)
    check(o32, ref32, f"{case} f16 in, f32 out")


@pytest.mark.parametrize("case", [(4, 64, 4096, 1024, True), (3, 200, 512, 384, False)])
def test_f16_unfused_and_my_id(agmm, case):
    P, m, k, n, rt = case
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=5, dtype="f16")
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, rt)
    unf, _ = _run(agmm, xs_cpu, y_cpu, rt, my_id=1, unfused=True)
    check(unf, ref32, f"{case} f16 unfused")
    for i in range(P):
        o, _ = _run(agmm, xs_cpu, y_cpu, rt, my_id=i)
        check(o, ref32, f"{case} f16 fused my_id={i}")


@pytest.mark.parametrize("name", ["c3_mid", "sweep_P8_m1000_rt", "c4_prefill"])
def test_f16_full_size(agmm, name):
    # every element of the mid-size workload and a ragged sweep point; on the
    # prefill-like workload one random row of every 128 output rows (every
    # row tile) and each shard's first, middle and last rows
    w = WORKLOADS[name]
    xs_cpu, y_cpu = make_inputs(w.P, w.m_per_device, w.k, w.n, w.rhs_transpose, w.dist, w.seed, dtype="f16")
    o, plan = _run(agmm, xs_cpu, y_cpu, w.rhs_transpose, my_id=w.my_id)
    if name != "c4_prefill":
        ref32, _ = oracle.agmm(xs_cpu, y_cpu, w.rhs_transpose)
        check_blocks(o, ref32, f"{name} f16 {plan.info()}")
        return
    rng = np.random.default_rng(3)
    rows = {int(t + rng.integers(0, min(128, w.M - t))) for t in range(0, w.M, 128)}
    for r in range(w.P):
        rows |= {r * w.m_per_device, r * w.m_per_device + w.m_per_device // 2, (r + 1) * w.m_per_device - 1}
    rows = sorted(rows)
    ref = oracle_rows(xs_cpu, y_cpu, w.rhs_transpose, rows)
    idx = torch.tensor(rows, device=o.device)
    check(o.index_select(0, idx), ref, f"{name} f16 {plan.info()}")
    assert bool(torch.isfinite(o.float()).all())


def test_f16_and_bf16_inputs_are_not_mixed(agmm):
    # the Python entry point takes the element type from the tensors
    xs_cpu, y_cpu = make_inputs(2, 16, 256, 128, False, seed=1, dtype="f16")
    xs = [x.cuda() for x in xs_cpu]
    with pytest.raises(ValueError):
        agmm.all_gather_matmul(xs, y_cpu.cuda().to(torch.bfloat16))
    o = agmm.all_gather_matmul(xs, y_cpu.cuda())
    torch.cuda.synchronize()
    assert o.dtype == torch.float16
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, False)
    check(o, ref32, "all_gather_matmul f16")
