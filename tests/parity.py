"""Shared helpers of the GPU parity tests: device placement with poisoned
guard rows, and the tolerance gate.

Tolerance (bf16 inputs, float32 accumulation):
  * float32 output mode: max |gpu - oracle_f32| <= 2e-2 and
    ||gpu - oracle_f32||_F / ||oracle_f32||_F <= 5e-3;
  * bf16 output: the same relative Frobenius bound, and per element
    |gpu - oracle_f32| <= max(2e-2, ulp_bf16(|oracle_f32|)).  A bf16 output
    cannot be closer to the float32 sum than half an ulp (0.03 for values in
    [8, 16)), and two correct float32 sums that straddle a rounding midpoint
    round one ulp apart, so the per-element bound is "2e-2 or one bf16 ulp".
  * fp16 output (fp16 inputs): the same gate with the fp16 ulp.  fp16 keeps
    11 significant bits, so below 32 the literal 2e-2 bound is the one that
    applies.
"""
import numpy as np
import torch

import oracle

MAX_ABS = 2e-2
REL_FRO = 5e-3
GUARD_ROWS = 3
BF16_NAN = 0x7FC0


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    a = np.abs(x.astype(np.float64))
    a = np.where(a < 2.0 ** -126, 2.0 ** -126, a)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def f16_ulp(x: np.ndarray) -> np.ndarray:
    a = np.abs(x.astype(np.float64))
    a = np.where(a < 2.0 ** -14, 2.0 ** -14, a)
    return 2.0 ** (np.floor(np.log2(a)) - 10)


def to_device_guarded(t: torch.Tensor, device="cuda"):
    """Copy a 2-D bf16 or fp16 tensor into a fresh allocation with NaN rows
    before and after it (0x7fc0 is a NaN in both types); returns (view of the
    payload, the whole buffer)."""
    rows, cols = t.shape
    buf = torch.empty((rows + 2 * GUARD_ROWS, cols), dtype=t.dtype, device=device)
    buf.view(torch.int16).fill_(BF16_NAN)
    view = buf[GUARD_ROWS:GUARD_ROWS + rows]
    view.copy_(t)
    return view, buf


def alloc_output_guarded(M, n, f32=False, device="cuda", f16=False):
    dt = torch.float32 if f32 else (torch.float16 if f16 else torch.bfloat16)
    buf = torch.full((M + 2 * GUARD_ROWS, n), float("nan"), dtype=dt, device=device)
    return buf[GUARD_ROWS:GUARD_ROWS + M], buf


def guards_intact(buf) -> bool:
    g = torch.cat([buf[:GUARD_ROWS], buf[-GUARD_ROWS:]])
    return bool(torch.isnan(g.float()).all())


def check(gpu_out: torch.Tensor, ref32: np.ndarray, tag: str = "") -> dict:
    g = gpu_out.float().cpu().numpy().astype(np.float64)
    r = ref32.astype(np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{tag}: non-finite outputs (unwritten rows?)"
    err = np.abs(g - r)
    fro = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))
    stats = {"max_abs": float(err.max()), "rel_fro": fro}
    assert fro <= REL_FRO, f"{tag}: relative Frobenius error {fro:.3e} > {REL_FRO}"
    if gpu_out.dtype == torch.float32:
        assert err.max() <= MAX_ABS, f"{tag}: max abs error {err.max():.3e} > {MAX_ABS}"
    else:
        ulp = f16_ulp(r) if gpu_out.dtype == torch.float16 else bf16_ulp(r)
        bound = np.maximum(MAX_ABS, ulp)
        bad = np.argwhere(err > bound)
        assert bad.size == 0, f"{tag}: {len(bad)} elements beyond max(2e-2, ulp); first {bad[:3].tolist()}"
    return stats


def check_blocks(gpu_out: torch.Tensor, ref32: np.ndarray, tag: str = "", rows_per_block: int = 1024) -> dict:
    """The gate of check() over every element of a large output, a block of
    rows at a time (bounded host memory): the relative Frobenius error is
    accumulated over all blocks, the per-element bound holds in each."""
    M = gpu_out.shape[0]
    assert ref32.shape == tuple(gpu_out.shape), (ref32.shape, tuple(gpu_out.shape))
    num = den = 0.0
    max_abs = 0.0
    for r0 in range(0, M, rows_per_block):
        r1 = min(M, r0 + rows_per_block)
        g = gpu_out[r0:r1].float().cpu().numpy().astype(np.float64)
        r = ref32[r0:r1].astype(np.float64)
        assert np.all(np.isfinite(g)), f"{tag}: non-finite outputs in rows [{r0}, {r1}) (unwritten rows?)"
        d = g - r
        num += float(np.sum(d * d))
        den += float(np.sum(r * r))
        err = np.abs(d)
        max_abs = max(max_abs, float(err.max()))
        if gpu_out.dtype == torch.float32:
            assert err.max() <= MAX_ABS, f"{tag}: max abs error {err.max():.3e} > {MAX_ABS} in rows [{r0}, {r1})"
        else:
            ulp = f16_ulp(r) if gpu_out.dtype == torch.float16 else bf16_ulp(r)
            bad = np.argwhere(err > np.maximum(MAX_ABS, ulp))
            assert bad.size == 0, (f"{tag}: {len(bad)} elements beyond max(2e-2, ulp) in rows [{r0}, {r1}); "
                                   f"first {(bad[:3] + [r0, 0]).tolist()}")
    fro = (num ** 0.5) / max(den ** 0.5, 1e-30)
    assert fro <= REL_FRO, f"{tag}: relative Frobenius error {fro:.3e} > {REL_FRO}"
    return {"max_abs": max_abs, "rel_fro": fro}


def oracle_rows(xs_cpu, y_cpu, rt, rows):
    """Oracle float32 sums of the selected output rows: the selected rows of
    the rank-order concatenation form a one-shard problem for the oracle."""
    sel = torch.cat(list(xs_cpu))[torch.tensor(list(rows))].contiguous()
    return oracle.agmm([sel], y_cpu, rt)[0]
