"""Run-time argument checks of the C ABI on a device: a workspace that
overlaps O, Y or a shard, a misaligned pointer or a bad my_id is rejected
with a status before anything is launched, so O keeps its poison."""
import pytest
import torch

from all_gather_gemm_agmm_gb300.inputs import make_inputs

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


def _status(agmm, fn):
    with pytest.raises(agmm.AgmmError) as err:
        fn()
    return err.value.status


@pytest.mark.parametrize("case", [(4, 64, 1024, 512, True), (3, 200, 512, 384, False)], ids=["swapped", "rows"])
def test_overlapping_workspace_is_rejected(agmm, case):
    P, m, k, n, rt = case
    xs_cpu, y_cpu = make_inputs(P, m, k, n, rt, seed=11)
    plan = agmm.Plan(P, m, k, n, rt)
    wsb = plan.workspace_bytes()
    wsu = plan.workspace_bytes(unfused=True)
    M = P * m
    # one arena holding O, Y and the shards, each 256-byte aligned
    o_elems, y_elems, x_elems = M * n, k * n, m * k
    pad = lambda e: (e + 127) // 128 * 128  # bf16 elements per 256 bytes
    arena = torch.zeros(pad(o_elems) + pad(y_elems) + P * pad(x_elems) + (wsu + 1) // 2 + 256,
                        dtype=torch.bfloat16, device="cuda")
    o = arena[:o_elems].view(M, n)
    y = arena[pad(o_elems):pad(o_elems) + y_elems].view(*y_cpu.shape)
    y.copy_(y_cpu)
    base = pad(o_elems) + pad(y_elems)
    xs = []
    for r in range(P):
        x = arena[base + r * pad(x_elems):base + r * pad(x_elems) + x_elems].view(m, k)
        x.copy_(xs_cpu[r])
        xs.append(x)
    o.view(torch.int16).fill_(0x7FC0)  # NaN poison
    torch.cuda.synchronize()

    def ws_at(t):  # a workspace view starting inside tensor t
        off = (t.data_ptr() - arena.data_ptr()) // 2
        return arena[off:].view(torch.uint8)

    for where in (o, y, xs[0], xs[-1]):
        ws = ws_at(where)
        assert _status(agmm, lambda: plan.run(xs, y, o, 0, ws)) == agmm.AGMM_ERR_INVALID_ARG
        assert _status(agmm, lambda: plan.run_unfused(xs, y, o, 0, ws)) == agmm.AGMM_ERR_INVALID_ARG
        xcat = torch.empty((M, k), dtype=torch.bfloat16, device="cuda")
        assert _status(agmm, lambda: plan.run_gather(xs, y, o, xcat, 0, ws)) == agmm.AGMM_ERR_INVALID_ARG
    assert "workspace overlaps" in agmm.load_library().agmm_last_error().decode()
    # a separate workspace is accepted (after a bad my_id and a misaligned one are not)
    ws_ok = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    assert _status(agmm, lambda: plan.run(xs, y, o, P, ws_ok)) == agmm.AGMM_ERR_INVALID_ARG  # my_id == P
    misaligned = ws_ok[8:]
    assert _status(agmm, lambda: plan.run(xs, y, o, 0, misaligned)) == agmm.AGMM_ERR_ALIGNMENT
    torch.cuda.synchronize()
    assert bool(torch.isnan(o.float()).all()), "a rejected call launched work"
    plan.run(xs, y, o, 0, ws_ok)
    plan.query_status(ws_ok)
    assert bool(torch.isfinite(o.float()).all())
