"""Tile configurations (agmm_tile_config_t) and the tuned table, on the CPU:
agmm_plan_preview honours each set field, rejects out-of-range values and
infeasible set fields, applies the precedence caller > environment > tuned
table > rules, and the committed table is the one the tuner writes from its
records."""
import ctypes
import json
import os

import pytest

import all_gather_gemm_agmm_gb300 as agmm
from all_gather_gemm_agmm_gb300 import tune
from all_gather_gemm_agmm_gb300.inputs import WORKLOADS

SMS = 152
RECORDS = os.path.join(agmm.PKG_DIR, "tuned_sm103.json")


@pytest.fixture(autouse=True)
def _library(agmm_lib, monkeypatch):
    for var in ("AGMM_PATH", "AGMM_CHUNKS", "AGMM_BN", "AGMM_CM", "AGMM_PAIR", "AGMM_STAGES", "AGMM_GROUP_M",
                "AGMM_STREAMK", "AGMM_ROWGROUPS", "AGMM_SPLITK", "AGMM_SWAP_DSMEM", "AGMM_TUNED"):
        monkeypatch.delenv(var, raising=False)
    return agmm_lib


def pv(P, m, k, n, rt=False, **cfg):
    return agmm.plan_preview(P, m, k, n, rt, num_sms=SMS, config=dict(cfg, tuned_table=False))


def status_of(P, m, k, n, rt=False, **cfg):
    with pytest.raises(agmm.AgmmError) as err:
        agmm.plan_preview(P, m, k, n, rt, num_sms=SMS, config=cfg)
    return err.value.status


def test_fields_are_honoured_on_row_tiles():
    P, m, k, n = 8, 1000, 1024, 2560  # ragged shards, 13 x 10 row tiles
    base = pv(P, m, k, n)
    assert base["path"] == 0 and base["tile_n"] == 256 and base["cluster_m"] == 2
    assert pv(P, m, k, n, tile_n=128)["tile_n"] == 128
    assert pv(P, m, k, n, cluster_m=1)["cluster_m"] == 1
    assert pv(P, m, k, n, cta_pair=True)["cta_pair"] == 1
    assert pv(P, m, k, n, stages=3)["stages"] == 3
    assert pv(P, m, k, n, group_m=4)["group_m"] == 4
    assert pv(P, m, k, n, chunks="whole")["whole_shards"] == 1
    assert pv(P, m, k, n, box_rows=32)["box_rows"] == 32
    assert base["stream_k_tiles"] > 0
    assert pv(P, m, k, n, stream_k=False)["stream_k_tiles"] == 0


def test_fields_are_honoured_on_swapped_tiles():
    w = WORKLOADS["c2_decode"]
    args = (w.P, w.m_per_device, w.k, w.n, w.rhs_transpose)
    base = pv(*args)
    assert base["path"] == 1
    assert pv(*args, path="rows")["path"] == 0
    assert pv(*args, row_groups=4)["row_groups"] == 4
    assert pv(*args, splits=3)["splits"] == 3
    assert pv(*args, dsmem_reduce=True)["dsmem_reduce"] == 1
    assert pv(*args, chunks="half")["whole_shards"] == 0
    assert pv(*args, box_rows=32, chunks="half")["box_rows"] == 32
    # a row-tile field is ignored on swapped tiles
    assert pv(*args, tile_n=256)["tile_n"] == base["tile_n"]
    # the rows path is chosen for a shape too tall for swapped tiles
    assert pv(8, 64, 512, 256)["path"] == 0


@pytest.mark.parametrize("cfg", [
    {"path": 3}, {"chunks": -1}, {"box_rows": 24}, {"box_rows": 256}, {"tile_n": 192}, {"cluster_m": 3},
    {"cta_pair": 3}, {"stream_k": -1}, {"stages": 1}, {"stages": 9}, {"group_m": -1}, {"row_groups": 3},
    {"row_groups": 512}, {"splits": 17}, {"splits": -2}, {"dsmem_reduce": 5}, {"tuned_table": 7},
])
def test_out_of_range_fields_are_invalid(cfg):
    assert status_of(2, 16, 256, 256, **cfg) == agmm.AGMM_ERR_INVALID_ARG


def test_infeasible_set_fields_are_unsupported():
    # more than 256 gathered rows cannot be swapped tiles
    assert status_of(8, 64, 512, 256, path="swap") == agmm.AGMM_ERR_UNSUPPORTED
    # tile_n must divide n
    assert status_of(8, 1000, 512, 384, path="rows", tile_n=256) == agmm.AGMM_ERR_UNSUPPORTED
    # a CTA pair needs a 2-CTA cluster, and a 2-CTA cluster is always a pair
    # (no copy is multicast to a cluster)
    assert status_of(8, 1000, 512, 512, cluster_m=1, cta_pair=True) == agmm.AGMM_ERR_UNSUPPORTED
    assert status_of(8, 1000, 512, 512, cluster_m=2, cta_pair=False) == agmm.AGMM_ERR_UNSUPPORTED
    # cta_pair off alone means one-CTA clusters
    assert pv(8, 1000, 512, 512, cta_pair=False)["cluster_m"] == 1
    # 2 chunks cannot make 4 non-empty row groups
    assert status_of(2, 16, 256, 256, chunks="whole", box_rows=16, row_groups=4) == agmm.AGMM_ERR_UNSUPPORTED


def test_raw_abi_config_and_null():
    lib = agmm.load_library()
    info = agmm.PlanInfo()
    tc = agmm.TileConfig()
    tc.path = 1  # row tiles
    assert lib.agmm_plan_preview(4, 64, 4096, 1024, 0, 1, ctypes.byref(tc), SMS, ctypes.byref(info)) == agmm.AGMM_OK
    assert info.path == 0 and info.config_source == 2
    assert lib.agmm_plan_preview(4, 64, 4096, 1024, 0, 1, None, SMS, ctypes.byref(info)) == agmm.AGMM_OK
    tc.splits = 99
    assert lib.agmm_plan_preview(4, 64, 4096, 1024, 0, 1, ctypes.byref(tc), SMS, ctypes.byref(info)) == \
        agmm.AGMM_ERR_INVALID_ARG
    # agmm_plan_config validates the shape and the config before any CUDA call
    h = ctypes.c_void_p()
    assert lib.agmm_plan_config(4, 64, 4096, 1024, 0, 1, ctypes.byref(tc), ctypes.byref(h)) == \
        agmm.AGMM_ERR_INVALID_ARG
    assert lib.agmm_plan_config(4, 64, 4096, 1024, 0, 1, None, None) == agmm.AGMM_ERR_INVALID_ARG


def test_precedence_caller_over_environment(monkeypatch):
    w = WORKLOADS["c2_decode"]
    args = (w.P, w.m_per_device, w.k, w.n, w.rhs_transpose)
    assert pv(*args)["config_source"] == 0
    monkeypatch.setenv("AGMM_ROWGROUPS", "4")
    info = agmm.plan_preview(*args, num_sms=SMS, config={"tuned_table": False})
    assert info["row_groups"] == 4 and info["config_source"] == 2
    assert pv(*args, row_groups=2)["row_groups"] == 2
    # an environment value that cannot hold is ignored, not an error
    monkeypatch.setenv("AGMM_ROWGROUPS", "64")
    assert pv(*args)["row_groups"] in (1, 2, 4, 8)
    monkeypatch.delenv("AGMM_ROWGROUPS")
    monkeypatch.setenv("AGMM_BN", "256")
    assert pv(8, 1000, 512, 384)["tile_n"] == 128


def test_config_dict_round_trip():
    cfg = {"path": "swap", "chunks": "whole", "box_rows": 64, "row_groups": 2, "splits": 6,
           "dsmem_reduce": False, "tuned_table": True}
    assert agmm.config_dict(agmm.tile_config(cfg)) == cfg
    with pytest.raises(ValueError):
        agmm.tile_config({"tile_q": 3})
    assert agmm.tile_config(None) is None


def _records():
    if not os.path.exists(RECORDS):
        pytest.skip("no tuning records committed")
    with open(RECORDS) as f:
        return json.load(f)["records"]


def test_committed_table_is_the_tuners_output(tmp_path):
    recs = _records()
    out = tmp_path / "table.inc"
    text = tune.emit(recs, str(out))
    with open(tune.TABLE_PATH) as f:
        assert f.read() == text


def test_table_entries_are_used_for_their_exact_shapes():
    recs = [r for r in _records() if r["tuned"]]
    for r in recs:
        args = (r["P"], r["m_per_device"], r["k"], r["n"], r["rhs_transpose"])
        got = agmm.plan_preview(*args, num_sms=SMS, f16=r["f16"])
        assert got["config_source"] == 1, r["name"]
        want = agmm.plan_preview(*args, num_sms=SMS, f16=r["f16"], config=dict(r["best"]["config"],
                                                                             tuned_table=False))
        for f in ("path", "box_rows", "whole_shards", "tile_n", "stages", "group_m", "row_groups", "cluster_m",
                  "cta_pair", "stream_k_tiles", "dsmem_reduce", "splits"):
            assert got[f] == want[f], (r["name"], f)
        # the switch turns the table off
        assert agmm.plan_preview(*args, num_sms=SMS, f16=r["f16"],
                                 config={"tuned_table": False})["config_source"] == 0
        # a neighbouring shape is not matched
        near = agmm.plan_preview(r["P"], r["m_per_device"] + 1, r["k"], r["n"], r["rhs_transpose"],
                                 num_sms=SMS, f16=r["f16"])
        assert near["config_source"] == 0


def test_table_entries_hold_only_winners():
    for r in _records():
        if r["tuned"]:
            assert r["best"]["us"] <= r["rules"]["us"] * (1 - tune.MARGIN), r["name"]


def test_candidates_are_distinct_and_start_with_the_rules():
    for name in ("c1_tiny", "c2_decode", "c3_mid", "sweep_P8_m8_nt"):
        w = WORKLOADS[name]
        cands = tune.candidates(w.P, w.m_per_device, w.k, w.n, w.rhs_transpose)
        assert cands[0] == {"tuned_table": False}
        keys = {tune._plan_key(agmm.plan_preview(w.P, w.m_per_device, w.k, w.n, w.rhs_transpose, num_sms=SMS,
                                                 config=c)) for c in cands}
        assert len(keys) == len(cands) > 3, name


def test_random_configs_plan_or_fail_cleanly():
    # any combination of fields either plans (and the plan keeps the planner's
    # invariants) or fails with a status, on random shapes
    import numpy as np

    rng = np.random.default_rng(99)
    choices = {
        "path": [0, 1, 2, "rows", "swap"], "chunks": [0, 1, 2], "box_rows": [0, 8, 16, 32, 64, 128],
        "tile_n": [0, 128, 256], "cluster_m": [0, 1, 2], "cta_pair": [None, True, False], "stages": [0, 2, 3, 5, 8],
        "group_m": [0, 1, 3, 8, 64], "stream_k": [None, True, False], "row_groups": [0, 1, 2, 4, 8],
        "splits": [0, 1, 2, 5, 16], "dsmem_reduce": [None, True, False], "tuned_table": [None, True, False],
    }
    planned = 0
    for _ in range(600):
        P = int(rng.integers(1, 9))
        m = int(rng.choice([1, 7, 16, 64, 100, 256, 1000]))
        k = 128 * int(rng.integers(1, 40))
        n = 128 * int(rng.integers(1, 30))
        cfg = {f: v[int(rng.integers(0, len(v)))] for f, v in choices.items() if rng.random() < 0.4}
        try:
            info = agmm.plan_preview(P, m, k, n, bool(rng.integers(0, 2)), num_sms=SMS, config=cfg)
        except agmm.AgmmError as e:
            assert e.status in (agmm.AGMM_ERR_INVALID_ARG, agmm.AGMM_ERR_UNSUPPORTED), (cfg, e)
            continue
        planned += 1
        assert 2 <= info["stages"] <= 8 and info["smem_bytes"] <= 232448, (cfg, info)
        assert info["box_rows"] in (8, 16, 32, 64, 128), (cfg, info)
        if info["path"] == 0:
            assert info["tile_n"] in (128, 256) and n % info["tile_n"] == 0, (cfg, info)
            assert info["cta_pair"] in (0, 1) and info["cta_pair"] == int(info["cluster_m"] == 2), (cfg, info)
        else:
            assert info["tile_n"] <= 256 and 1 <= info["splits"] <= 16, (cfg, info)
    assert planned > 200
