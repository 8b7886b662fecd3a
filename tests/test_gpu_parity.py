"""GPU parity: the sm_103a kernels (through the C ABI) against the CPU oracle
on the same seeded inputs."""
import os

import pytest
import torch

import oracle
from all_gather_gemm_agmm_gb300.inputs import SWEEP, WORKLOADS, make_inputs

from parity import alloc_output_guarded, check, check_blocks, guards_intact, to_device_guarded

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


def _run(agmm, xs_cpu, y_cpu, rt, my_id, f32=False, unfused=False, plan=None):
    P = len(xs_cpu)
    m, k = xs_cpu[0].shape
    n = y_cpu.shape[0] if rt else y_cpu.shape[1]
    xs = [to_device_guarded(x)[0] for x in xs_cpu]
    y, _ = to_device_guarded(y_cpu)
    o, obuf = alloc_output_guarded(P * m, n, f32)
    plan = plan or agmm.Plan(P, m, k, n, rt, f32)
    ws = plan.new_workspace(unfused)
    (plan.run_unfused if unfused else plan.run)(xs, y, o, my_id, ws)
    plan.query_status(ws)
    torch.cuda.synchronize()
    assert guards_intact(obuf), "a store landed outside O"
    return o, plan


# Small and mid cases the oracle finishes in seconds: several tiles, ragged
# tails, odd shards, both layouts, both paths.
SMALL = [
    # P, m_pd, k, n, rt, dist
    (2, 16, 256, 128, False, "uniform"),   # the tiny uniform workload
    (4, 64, 4096, 1024, True, "normal"),   # the decode-like workload, full size
    (8, 8, 1024, 256, False, "normal"),
    (3, 5, 128, 128, True, "normal"),
    (1, 1, 128, 128, False, "normal"),
    (2, 128, 512, 384, True, "normal"),
    (3, 200, 512, 384, False, "normal"),   # rows path, ragged halves of 100
    (2, 300, 256, 512, True, "normal"),    # rows path, n tile 256
    (5, 77, 384, 256, False, "uniform"),   # rows path, odd shards
    (8, 130, 256, 640, True, "normal"),    # rows path, n 640 = 5 x 128
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "P{}_m{}_k{}_n{}_{}".format(*c[:4], "rt" if c[4] else "nt"))
def test_parity_small(agmm, case):
    P, m, k, n, rt, dist = case
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, dist=dist, seed=0)
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, rt)
    o, plan = _run(agmm, xs_cpu, y_cpu, rt, my_id=P - 1)
    check(o, ref32, f"{case} bf16 {plan.info()}")
    o32, _ = _run(agmm, xs_cpu, y_cpu, rt, my_id=0, f32=True)
    check(o32, ref32, f"{case} f32")


@pytest.mark.parametrize("case", [(3, 200, 512, 384, False), (4, 64, 1024, 256, True), (5, 9, 256, 128, False)])
def test_result_independent_of_my_id(agmm, case):
    P, m, k, n, rt = case
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=1)
    outs = [_run(agmm, xs_cpu, y_cpu, rt, my_id=i)[0] for i in range(P)]
    for i in range(1, P):
        assert torch.equal(outs[0].view(torch.int16), outs[i].view(torch.int16)), f"my_id {i} differs"


@pytest.mark.parametrize("case", [(4, 64, 4096, 1024, True), (3, 200, 512, 384, False), (2, 300, 256, 512, True)])
def test_unfused_matches(agmm, case):
    P, m, k, n, rt = case
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=2)
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, rt)
    fused, _ = _run(agmm, xs_cpu, y_cpu, rt, my_id=1)
    unf, _ = _run(agmm, xs_cpu, y_cpu, rt, my_id=1, unfused=True)
    check(unf, ref32, f"{case} unfused")
    check(fused, ref32, f"{case} fused")


@pytest.mark.parametrize("force_rows", [True])
def test_rows_path_on_small_m(agmm, force_rows, monkeypatch):
    # The planner sends small problems to the swapped tiles; force the row
    # tiles (box heights 8 and 16) to cover them too.
    monkeypatch.setenv("AGMM_PATH", "0")
    for (P, m, k, n, rt) in [(2, 16, 256, 128, False), (8, 8, 512, 256, True), (3, 5, 256, 256, False)]:
        xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=3)
        ref32, _ = oracle.agmm(xs_cpu, y_cpu, rt)
        o, plan = _run(agmm, xs_cpu, y_cpu, rt, my_id=P - 1)
        assert plan.info()["path"] == 0
        check(o, ref32, f"forced rows {P},{m}")


# Every element of the full-size workloads against the oracle: the mid-size
# and prefill-like workloads and all 30 sweep points (P in {2, 4, 8} x
# m_per_device in {8, 32, 128, 1000, 4096} x both Y layouts), each with its
# own my_id and the launch configuration the benchmark times.
FULL = ["c3_mid", "c4_prefill"] + [w.name for w in SWEEP]


@pytest.mark.parametrize("name", FULL)
def test_parity_full_size(agmm, name):
    w = WORKLOADS[name]
    xs_cpu, y_cpu = make_inputs(w.P, w.m_per_device, w.k, w.n, w.rhs_transpose, w.dist, w.seed)
    o, plan = _run(agmm, xs_cpu, y_cpu, w.rhs_transpose, my_id=w.my_id)
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, w.rhs_transpose)
    check_blocks(o, ref32, f"{name} {plan.info()}")


@pytest.mark.parametrize("streamk", ["0", "1"])
def test_stream_k_split(agmm, streamk, monkeypatch):
    # Tiles beyond the last whole wave are spread over the clusters by k
    # blocks; owners add the contributors' float32 partials in k order.
    monkeypatch.setenv("AGMM_STREAMK", streamk)
    for (P, m, k, n, rt) in [(5, 77, 1024, 256, False), (3, 200, 2048, 384, True), (8, 260, 768, 1280, False)]:
        xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=4)
        ref32, _ = oracle.agmm(xs_cpu, y_cpu, rt)
        o, plan = _run(agmm, xs_cpu, y_cpu, rt, my_id=1)
        check(o, ref32, f"stream-k {streamk} {plan.info()}")
        # a second run reuses the counters the owners reset
        o2, _ = _run(agmm, xs_cpu, y_cpu, rt, my_id=1, plan=plan)
        assert torch.equal(o.view(torch.int16), o2.view(torch.int16))


@pytest.mark.parametrize("case", [(3, 200, 1024, 512, False), (5, 300, 512, 256, True), (8, 130, 256, 640, True),
                                  (4, 256, 768, 768, False)])
def test_cluster_variants(agmm, case, monkeypatch):
    # Row tiles either one CTA per cluster, or clusters of two that multiply
    # as one cta_group::2 MMA per pair (each CTA loads and holds half the Y
    # tile; no copy is multicast).  Both meet the oracle tolerance; odd
    # row-tile counts exercise an idle second CTA.  A two-CTA cluster without
    # the pair is not a plan.
    P, m, k, n, rt = case
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=6)
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, rt)
    monkeypatch.setenv("AGMM_STREAMK", "0")
    for name, cm, pair in (("single", "1", "0"), ("pair", "2", "1")):
        monkeypatch.setenv("AGMM_CM", cm)
        monkeypatch.setenv("AGMM_PAIR", pair)
        o, plan = _run(agmm, xs_cpu, y_cpu, rt, my_id=P - 1)
        info = plan.info()
        assert info["cluster_m"] == int(cm) and info["cta_pair"] == int(pair == "1"), info
        check(o, ref32, f"{name} {info}")
    with pytest.raises(agmm.AgmmError) as err:
        agmm.Plan(P, m, k, n, rt, config={"path": "rows", "cluster_m": 2, "cta_pair": False})
    assert err.value.status == agmm.AGMM_ERR_UNSUPPORTED


@pytest.mark.parametrize("mode", ["half", "whole"])
@pytest.mark.parametrize("case", [(2, 16, 256, 128, False, "uniform"), (4, 64, 1024, 1024, True, "normal"),
                                  (8, 8, 512, 256, False, "normal"), (3, 13, 256, 256, True, "normal"),
                                  (8, 128, 512, 512, True, "normal"), (3, 200, 512, 384, False, "normal")],
                         ids=lambda c: "P{}_m{}".format(c[0], c[1]) if isinstance(c, tuple) else c)
def test_chunking_modes(agmm, case, mode, monkeypatch):
    # Half-shard chunks follow the ring's left/right split; whole-shard chunks
    # follow the ring's first-visit shard order.  Both give the same product.
    monkeypatch.setenv("AGMM_CHUNKS", mode)
    P, m, k, n, rt, dist = case
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, dist=dist, seed=8)
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, rt)
    o, plan = _run(agmm, xs_cpu, y_cpu, rt, my_id=P // 2)
    assert plan.info()["whole_shards"] == (mode == "whole")
    check(o, ref32, f"{mode} {plan.info()}")


@pytest.mark.parametrize("case", [(4, 64, 1024, 512, True), (5, 40, 512, 256, False), (3, 13, 768, 384, True),
                                  (8, 32, 512, 256, False)],
                         ids=lambda c: "P{}_m{}_k{}".format(c[0], c[1], c[2]))
def test_swap_row_groups(agmm, case, monkeypatch):
    # The swapped path may divide the ring-ordered chunks into row groups,
    # each its own MMA N.  With the k splits fixed, every output element is
    # reduced in the same order whatever the grouping, so the groupings agree
    # bitwise; both reduction routes (device memory, distributed shared
    # memory) meet the oracle tolerance.  Odd chunk counts leave a short last
    # group.
    P, m, k, n, rt = case
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=9)
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, rt)
    monkeypatch.setenv("AGMM_PATH", "1")
    monkeypatch.setenv("AGMM_SPLITK", "4")
    outs = {}
    used_dsmem = 0
    for dsmem in ("0", "1"):
        monkeypatch.setenv("AGMM_SWAP_DSMEM", dsmem)
        for groups in ("1", "2", "4"):
            monkeypatch.setenv("AGMM_ROWGROUPS", groups)
            o, plan = _run(agmm, xs_cpu, y_cpu, rt, my_id=P - 1)
            info = plan.info()
            assert info["path"] == 1
            if info["row_groups"] != int(groups):
                continue  # that many groups would leave one empty
            check(o, ref32, f"groups={groups} dsmem={dsmem} {info}")
            assert info["splits"] == 4, info  # both routes keep the k splits
            outs[(dsmem, groups)] = o
            used_dsmem += info["dsmem_reduce"]
    base = outs[("0", "1")]
    for key, o in outs.items():
        assert torch.equal(base.view(torch.int16), o.view(torch.int16)), key
    assert used_dsmem > 0  # the distributed-shared-memory route ran


@pytest.mark.parametrize("case", [(4, 64, 1024, 512, True), (3, 13, 768, 384, False), (8, 8, 2048, 256, True)],
                         ids=lambda c: "P{}_m{}_k{}".format(c[0], c[1], c[2]))
def test_swap_reduction_routes(agmm, case):
    # Swapped tiles reduce their k splits one of three ways: no split (the
    # CTA stores its own accumulator), through an L2-resident workspace, or
    # by bulk copies into the owners' shared memory.  Every route meets the
    # oracle in bf16 and float32 output; with the same splits the two
    # cross-CTA routes agree bitwise (same rank-order sums).
    P, m, k, n, rt = case
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=21)
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, rt)
    for splits in (1, 5, 8, 16):
        outs = {}
        for dsmem in (False, True):
            cfg = {"path": "swap", "splits": splits, "dsmem_reduce": dsmem, "tuned_table": False}
            try:
                plan = agmm.Plan(P, m, k, n, rt, config=cfg)
            except agmm.AgmmError as e:
                assert e.status == agmm.AGMM_ERR_UNSUPPORTED, e
                continue
            info = plan.info()
            assert info["path"] == 1
            for f32 in (False, True):
                pl = plan if not f32 else agmm.Plan(P, m, k, n, rt, out_f32=True, config=cfg)
                o, _ = _run(agmm, xs_cpu, y_cpu, rt, my_id=P - 1, f32=f32, plan=pl)
                check(o, ref32, f"splits={splits} dsmem={dsmem} f32={f32} {pl.info()}")
                if not f32:
                    outs[(dsmem, info["splits"], info["dsmem_reduce"])] = o
        same_split = {}
        for (dsmem, s, used), o in outs.items():
            same_split.setdefault(s, []).append(o)
        for s, os_ in same_split.items():
            for o in os_[1:]:
                assert torch.equal(os_[0].view(torch.int16), o.view(torch.int16)), (case, s)


@pytest.mark.parametrize("case", [(3, 200, 1024, 512, False), (4, 128, 1280, 512, True), (8, 130, 768, 1280, True)],
                         ids=lambda c: "P{}_m{}_n{}".format(c[0], c[1], c[3]))
def test_row_tiles_k_blocks_per_stage(agmm, case, monkeypatch):
    # Row tiles stage one or two k blocks per pipeline step (the planner takes
    # two for 128-wide tiles); both meet the oracle and, with the same tiles
    # and k partition, agree bitwise (the MMAs accumulate in the same order).
    P, m, k, n, rt = case
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=23)
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, rt)
    for bn in ("128", "256"):
        if int(n) % int(bn):
            continue
        monkeypatch.setenv("AGMM_BN", bn)
        outs = []
        for atoms in ("1", "2"):
            monkeypatch.setenv("AGMM_ATOMS", atoms)
            o, plan = _run(agmm, xs_cpu, y_cpu, rt, my_id=1)
            assert plan.info()["path"] == 0 and plan.info()["tile_n"] == int(bn)
            assert plan.info()["k_blocks_per_stage"] == int(atoms)
            check(o, ref32, f"BN {bn} atoms {atoms} {plan.info()}")
            outs.append(o)
        assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16)), (case, bn)
