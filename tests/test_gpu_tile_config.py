"""GPU parity of plans built from explicit tile configurations
(agmm_plan_config): every variant the tuner may put in the tuned table must
meet the same parity gate against the oracle, and the plan must report the
configuration it was given."""
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


def _run_config(agmm, shape, cfg, seed):
    P, m, k, n, rt = shape
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=seed)
    ref32, _ = oracle.agmm(xs_cpu, y_cpu, rt)
    xs = [to_device_guarded(x)[0] for x in xs_cpu]
    y, _ = to_device_guarded(y_cpu)
    o, obuf = alloc_output_guarded(P * m, n)
    plan = agmm.Plan(P, m, k, n, rt, config=cfg)
    ws = plan.new_workspace()
    torch.cuda.synchronize()
    plan.run(xs, y, o, P - 1, ws)
    plan.query_status(ws)
    torch.cuda.synchronize()
    assert guards_intact(obuf), "a store landed outside O"
    check(o, ref32, f"{shape} {cfg} {plan.info()}")
    return plan.info()


ROWS = (3, 200, 512, 768, False)  # 5 row tiles (ragged halves), 3 n tiles of 256
SWAP = (4, 64, 1024, 512, True)


@pytest.mark.parametrize("cfg", [
    {"path": "rows", "tile_n": 128},
    {"path": "rows", "cluster_m": 1},
    {"path": "rows", "cta_pair": True},
    {"path": "rows", "stream_k": False, "group_m": 2},
    {"path": "rows", "cluster_m": 1, "stream_k": True},  # one-CTA clusters: cooperative launch
    {"path": "rows", "chunks": "whole", "box_rows": 64, "stages": 3},
], ids=str)
def test_row_tile_configs(agmm, cfg):
    info = _run_config(agmm, ROWS, cfg, seed=31)
    assert info["path"] == 0 and info["config_source"] == 2
    if "tile_n" in cfg:
        assert info["tile_n"] == cfg["tile_n"]
    if "cluster_m" in cfg:
        assert info["cluster_m"] == cfg["cluster_m"]
    if cfg.get("cta_pair"):
        assert info["cta_pair"] == 1
    if "stages" in cfg:
        assert info["stages"] == cfg["stages"]
    if cfg.get("stream_k"):
        assert info["stream_k_tiles"] > 0


@pytest.mark.parametrize("cfg", [
    {"path": "swap", "row_groups": 1, "splits": 2},
    {"path": "swap", "row_groups": 2, "splits": 4},
    {"path": "swap", "row_groups": 4, "splits": 3, "chunks": "half"},
    {"path": "swap", "dsmem_reduce": True, "splits": 4},
    {"path": "swap", "chunks": "half", "box_rows": 16},
], ids=str)
def test_swapped_tile_configs(agmm, cfg):
    info = _run_config(agmm, SWAP, cfg, seed=32)
    assert info["path"] == 1
    if "row_groups" in cfg:
        assert info["row_groups"] == cfg["row_groups"]
    if "box_rows" in cfg:
        assert info["box_rows"] == cfg["box_rows"]
    assert 1 <= info["splits"] <= cfg.get("splits", 16)


def test_infeasible_config_fails_before_launch(agmm):
    with pytest.raises(agmm.AgmmError) as err:
        agmm.Plan(8, 64, 512, 256, False, config={"path": "swap"})
    assert err.value.status == agmm.AGMM_ERR_UNSUPPORTED


def test_random_configs_match_oracle(agmm):
    # seeded random (shape, configuration) pairs the planner accepts: every
    # one meets the parity gate, with nothing stored outside O
    import numpy as np

    rng = np.random.default_rng(123)
    choices = {
        "path": ["rows", "swap"], "chunks": ["half", "whole"], "box_rows": [8, 16, 32, 64, 128],
        "tile_n": [128, 256], "cluster_m": [1, 2], "cta_pair": [True, False], "stages": [2, 3, 8],
        "group_m": [1, 3, 8], "stream_k": [True, False], "row_groups": [1, 2, 4], "splits": [1, 2, 3, 6],
        "dsmem_reduce": [True, False],
    }
    ran = 0
    for trial in range(40):
        P = int(rng.integers(1, 6))
        m = int(rng.choice([5, 16, 40, 77, 130]))
        k = 128 * int(rng.integers(1, 6))
        n = 256 * int(rng.integers(1, 3))
        rt = bool(rng.integers(0, 2))
        cfg = {f: v[int(rng.integers(0, len(v)))] for f, v in choices.items() if rng.random() < 0.5}
        cfg["tuned_table"] = False
        try:
            agmm.plan_preview(P, m, k, n, rt, config=cfg)
        except agmm.AgmmError:
            continue  # a combination this shape cannot hold
        xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=200 + trial)
        ref32, _ = oracle.agmm(xs_cpu, y_cpu, rt)
        xs = [to_device_guarded(x)[0] for x in xs_cpu]
        y, _ = to_device_guarded(y_cpu)
        o, obuf = alloc_output_guarded(P * m, n)
        plan = agmm.Plan(P, m, k, n, rt, config=cfg)
        ws = plan.new_workspace()
        torch.cuda.synchronize()
        plan.run(xs, y, o, int(rng.integers(0, P)), ws)
        plan.query_status(ws)
        torch.cuda.synchronize()
        assert guards_intact(obuf), (P, m, k, n, rt, cfg)
        check(o, ref32, f"{(P, m, k, n, rt)} {cfg} {plan.info()}")
        ran += 1
    assert ran >= 15
