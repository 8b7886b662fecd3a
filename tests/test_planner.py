"""Host-side planning, on the CPU: agmm_plan_preview runs the planner's tile
choice without CUDA.  Pins the plans of the named workloads (the choices the
GPU runs were measured with) and checks invariants of the planner on random
shapes, including agreement with agmm_ring_chunks."""
import ctypes

import numpy as np
import pytest

import all_gather_gemm_agmm_gb300 as agmm
from all_gather_gemm_agmm_gb300.inputs import WORKLOADS

MAX_DYN_SMEM = 232448  # bytes of dynamic shared memory a CTA may use
SMS = 152


@pytest.fixture(autouse=True)
def _library(agmm_lib):
    # built in-tree (nvcc cross-compiles) before any preview call
    return agmm_lib


def preview(w, **kw):
    # the planner's own rules: the tuned table is switched off
    return agmm.plan_preview(w.P, w.m_per_device, w.k, w.n, w.rhs_transpose, num_sms=SMS,
                             config={"tuned_table": False}, **kw)


# (path, box_rows, whole_shards, chunks, tile_n, stages, row_groups, split bound,
# k blocks per stage);
# row tiles in two-CTA clusters multiply as CTA pairs (half the Y tile per
# CTA), hence 7 stages of 32 KiB at 256-wide tiles; 128-wide row tiles and
# swapped tiles stage two k blocks at a time
PINNED = {
    "c1_tiny": (1, 16, 1, 2, 32, 5, 2, 4, 2),
    "c2_decode": (1, 64, 1, 4, 128, 3, 2, 9, 2),
    "c3_mid": (0, 128, 0, 16, 256, 7, 1, 1, 1),
    "c4_prefill": (0, 128, 0, 128, 256, 7, 1, 1, 1),
    "sweep_P8_m8_nt": (1, 8, 1, 8, 64, 4, 1, 7, 2),
    "sweep_P2_m1000_nt": (0, 128, 0, 16, 256, 7, 1, 1, 1),
    # 128-wide (256-wide gives 20 cluster tiles), two k blocks per stage: 4 stages of 2 x 24 KiB
    "sweep_P4_m128_rt": (0, 128, 1, 4, 128, 4, 1, 1, 2),
}


@pytest.mark.parametrize("name", sorted(PINNED))
def test_pinned_workload_plans(name):
    info = preview(WORKLOADS[name])
    got = (info["path"], info["box_rows"], info["whole_shards"], info["chunks"], info["tile_n"], info["stages"],
           info["row_groups"], info["splits"], info["k_blocks_per_stage"])
    assert got == PINNED[name], (name, info)


def _ring_count(P, m, box, whole):
    lib = agmm.load_library()
    n = ctypes.c_int64()
    st = lib.agmm_ring_chunks(P, m, 0, box, whole, None, None, None, None, 0, ctypes.byref(n))
    assert st == agmm.AGMM_OK
    return n.value


def test_planner_invariants_random_shapes():
    rng = np.random.default_rng(2024)
    for _ in range(400):
        P = int(rng.integers(1, 9))
        m = int(rng.choice([1, 3, 8, 13, 32, 64, 77, 128, 200, 1000, 4096]))
        k = 128 * int(rng.integers(1, 80))
        n = 128 * int(rng.integers(1, 60))
        rt = bool(rng.integers(0, 2))
        f16 = bool(rng.integers(0, 2))
        info = agmm.plan_preview(P, m, k, n, rt, num_sms=SMS, f16=f16)
        tag = (P, m, k, n, rt, info)
        assert 2 <= info["stages"] <= 8, tag
        assert info["smem_bytes"] <= MAX_DYN_SMEM, tag
        box = info["box_rows"]
        assert box in (8, 16, 32, 64, 128), tag
        # the planner's chunk count is the ring schedule's
        assert info["chunks"] == _ring_count(P, m, box, info["whole_shards"]), tag
        padded = info["chunks"] * box
        assert padded >= P * m, tag  # every gathered row lies in some chunk
        if info["path"] == 1:
            # swapped tiles: all gathered rows in MMA N <= 256, n tiles of 128
            G = info["row_groups"]
            cpg = -(-info["chunks"] // G)
            assert padded <= 256, tag
            assert (G - 1) * cpg < info["chunks"], tag  # no empty row group
            assert info["tile_n"] % 32 == 0 and cpg * box <= info["tile_n"] <= 256, tag
            assert 1 <= info["splits"] <= min(16, k // 64), tag
            assert info["num_tiles"] == n // 128, tag
        else:
            assert info["tile_n"] in (128, 256) and n % info["tile_n"] == 0, tag
            assert info["splits"] == 1 and info["row_groups"] == 1, tag


def test_small_problems_take_swapped_tiles():
    # whenever some chunking of the gathered rows fits one MMA N, the swapped
    # tiles are chosen (they read Y from device memory once)
    for P, m in [(1, 1), (2, 16), (4, 64), (8, 32), (3, 13), (2, 128)]:
        assert agmm.plan_preview(P, m, 1024, 512, False)["path"] == 1, (P, m)
    for P, m in [(2, 200), (8, 64), (4, 1000)]:
        assert agmm.plan_preview(P, m, 1024, 512, False)["path"] == 0, (P, m)


def test_environment_overrides(monkeypatch):
    w = WORKLOADS["c2_decode"]
    monkeypatch.setenv("AGMM_PATH", "0")
    assert preview(w)["path"] == 0
    monkeypatch.delenv("AGMM_PATH")
    monkeypatch.setenv("AGMM_ROWGROUPS", "4")
    monkeypatch.setenv("AGMM_SPLITK", "4")
    info = preview(w)
    assert (info["row_groups"], info["splits"]) == (4, 4)
    monkeypatch.setenv("AGMM_CHUNKS", "half")
    assert preview(w)["whole_shards"] == 0


def test_preview_argument_errors():
    lib = agmm.load_library()
    info = agmm.PlanInfo()
    assert lib.agmm_plan_preview(2, 16, 256, 128, 0, 0, None, 0, ctypes.byref(info)) == agmm.AGMM_ERR_INVALID_ARG
    assert lib.agmm_plan_preview(2, 16, 256, 128, 0, 0, None, 152, None) == agmm.AGMM_ERR_INVALID_ARG
    assert lib.agmm_plan_preview(2, 16, 200, 128, 0, 0, None, 152, ctypes.byref(info)) == agmm.AGMM_ERR_INVALID_ARG
    assert lib.agmm_plan_preview(9, 16, 256, 128, 0, 0, None, 152, ctypes.byref(info)) == agmm.AGMM_ERR_INVALID_ARG
    assert lib.agmm_plan_preview(2, 16, 256, 128, 5, 0, None, 152, ctypes.byref(info)) == agmm.AGMM_ERR_INVALID_ARG


def _tmem_cols(info):
    if info["path"] == 0:
        return 2 * info["tile_n"]  # two accumulators of tile_n columns
    c = 32
    while c < info["tile_n"]:
        c *= 2
    return c


@pytest.mark.parametrize("stages", ["2", "3", "8"])
def test_resident_ctas_fit_tensor_memory(stages, monkeypatch):
    # tcgen05.alloc waits for free columns: the CTAs that fit on one SM by
    # shared memory (228 KiB, 1 KiB reserved per CTA) must fit in its 512
    # TMEM columns together, even when fewer pipeline stages shrink a CTA
    monkeypatch.setenv("AGMM_STAGES", stages)
    rng = np.random.default_rng(7)
    for _ in range(150):
        P = int(rng.integers(1, 9))
        m = int(rng.choice([1, 8, 16, 64, 128, 300, 2048]))
        k = 128 * int(rng.integers(1, 40))
        n = 256 * int(rng.integers(1, 20))
        info = agmm.plan_preview(P, m, k, n, bool(rng.integers(0, 2)), num_sms=SMS)
        resident = 233472 // (info["smem_bytes"] + 1024)
        assert 1 <= resident and resident * _tmem_cols(info) <= 512, (P, m, k, n, info)


def test_stream_k_fill_rule():
    # A ragged last wave of cluster tiles goes to stream-K unless it already
    # fills two thirds of the clusters (76 CTA pairs on 152 SMs); stream-K set
    # on by the configuration applies whatever the fill.
    tt = {"tuned_table": False}
    cases = {"c4_quarter": (448, 0), "c4_prefill": (1792, 44), "c3_mid": (112, 36),
             "sweep_P8_m4096_nt": (1280, 0), "sweep_P4_m1000_nt": (160, 84)}
    for name, (tiles, sk) in cases.items():
        w = WORKLOADS[name]
        info = agmm.plan_preview(w.P, w.m_per_device, w.k, w.n, w.rhs_transpose, num_sms=SMS, config=tt)
        assert (info["num_tiles"], info["stream_k_tiles"]) == (tiles, sk), name
        ragged = tiles % (SMS // 2)
        assert (sk == 0) == (ragged == 0 or 3 * ragged >= 2 * (SMS // 2)), name
    w = WORKLOADS["c4_quarter"]
    on = agmm.plan_preview(w.P, w.m_per_device, w.k, w.n, w.rhs_transpose, num_sms=SMS,
                           config={"tuned_table": False, "stream_k": True})
    assert on["stream_k_tiles"] == 448 % (SMS // 2)
    off = agmm.plan_preview(w.P, w.m_per_device, w.k, w.n, w.rhs_transpose, num_sms=SMS,
                            config={"tuned_table": False, "stream_k": False})
    assert off["stream_k_tiles"] == 0
