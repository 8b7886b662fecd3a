"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

Each pin is a plain function of a loaded oracle library, so that the mutation
test at the end can run the same pins against copies of the oracle with a
planted mistake and show that every mistake is caught.

Pins:
  * bf16 rounding: hand-worked bit patterns (tests/golden/bf16_rounding.json)
  * fp16 rounding and decoding: hand-worked bit patterns
    (tests/golden/f16_rounding.json), PyTorch's casts, and the fp16 product
    by the same invariants as the bf16 one
    and agreement with PyTorch's float32 -> bfloat16 cast (a library routine).
  * a hand-worked example (tests/golden/hand_example.json), both layouts.
  * P = 1 reduces to a plain matmul: checked against torch.matmul in float64
    within the float32 dot-product error bound gamma_k * sum |x||y|.
  * identity embedding: Y = [I_n; 0] returns the gathered X exactly.
  * shard isolation and placement: only shard r nonzero -> only row block r
    nonzero, equal to shard r alone times Y.
  * shard permutation permutes the output row blocks.
  * scaling Y by 2 scales O by exactly 2.
  * brute force with exact rationals on tiny shapes, then exact RNE to bf16.
  * bf16 decoding: all 65536 patterns against the binary32 upper-half rule.
"""
from __future__ import annotations

import ctypes
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from all_gather_gemm_agmm_gb300.inputs import make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U = 2.0 ** -24  # unit roundoff of float32


def gamma(k: int) -> float:
    return k * U / (1.0 - k * U)


def _f32(bits):
    return oracle.bits_to_f32(bits)


def _cat_f64(xs):
    return np.concatenate([oracle.bits_to_f32(oracle.as_bf16_bits(x)).astype(np.float64) for x in xs])


def _ycan_f64(y, rt):
    yf = oracle.bits_to_f32(oracle.as_bf16_bits(y)).astype(np.float64)
    return yf.T if rt else yf


def _bf16_from_floats(a):
    return torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


# ----------------------------------------------------------------------------- pins

def pin_bf16_golden(lib):
    with open(os.path.join(GOLDEN, "bf16_rounding.json")) as f:
        cases = json.load(f)["cases"]
    for f32hex, bf16hex, why in cases:
        f = np.array([int(f32hex, 16)], dtype=np.uint32).view(np.float32)
        got = int(oracle.f32_to_bf16_bits(f, lib)[0])
        assert got == int(bf16hex, 16), (f32hex, hex(got), why)
    # NaN in -> NaN out (payload is not pinned)
    for nan_bits in (0x7FC00000, 0x7F800001, 0xFFC00001):
        f = np.array([nan_bits], dtype=np.uint32).view(np.float32)
        got = int(oracle.f32_to_bf16_bits(f, lib)[0])
        assert (got & 0x7F80) == 0x7F80 and (got & 0x007F) != 0, hex(got)


def pin_bf16_vs_torch(lib):
    rng = np.random.default_rng(1234)
    bits = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    f = f[np.isfinite(f)]
    # add values that sit exactly on ties
    ties = (rng.integers(0, 2 ** 16, size=20_000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    tf = ties.view(np.float32)
    f = np.concatenate([f, tf[np.isfinite(tf)]])
    ours = oracle.f32_to_bf16_bits(f, lib)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(hex(int(f.view(np.uint32)[i])), hex(int(ours[i])), hex(int(ref[i]))) for i in bad[:5]]


def pin_hand_example(lib):
    with open(os.path.join(GOLDEN, "hand_example.json")) as fh:
        g = json.load(fh)
    xs = [_bf16_from_floats(s) for s in g["x_shards"]]
    y_kn = _bf16_from_floats(g["y_kn"])
    exp = np.asarray(g["expected"], dtype=np.float32)
    o32, o16 = oracle.agmm(xs, y_kn, False, lib=lib)
    assert np.array_equal(o32, exp), o32
    assert np.array_equal(_f32(o16), exp)
    o32t, _ = oracle.agmm(xs, y_kn.T.contiguous(), True, lib=lib)
    assert np.array_equal(o32t, exp), o32t


def pin_plain_matmul_p1(lib):
    for (m, k, n, rt, dist) in [(7, 64, 24, False, "uniform"), (5, 256, 40, True, "normal"),
                                (33, 130, 17, False, "normal"), (16, 512, 128, True, "uniform")]:
        xs, y = make_inputs(1, m, k, n, rt, dist=dist, seed=7)
        o32, _ = oracle.agmm(xs, y, rt, lib=lib)
        a = _cat_f64(xs)
        b = _ycan_f64(y, rt)
        ref = (torch.from_numpy(a) @ torch.from_numpy(b)).numpy()
        bound = gamma(k) * (np.abs(a) @ np.abs(b)) + 1e-30
        err = np.abs(o32.astype(np.float64) - ref)
        assert np.all(err <= bound), (m, k, n, rt, float((err / bound).max()))
        # the dot products are not trivially exact: some rounding did happen
        assert np.any(err > 0) or dist == "none"


def pin_identity_embedding(lib):
    for rt in (False, True):
        P, m, k, n = 3, 5, 48, 32
        xs, _ = make_inputs(P, m, k, n, rt, dist="normal", seed=3)
        eye = torch.zeros((k, n), dtype=torch.float32)
        eye[:n, :n] = torch.eye(n)
        y = (eye.T.contiguous() if rt else eye).to(torch.bfloat16)
        o32, o16 = oracle.agmm(xs, y, rt, lib=lib)
        xcat = np.concatenate([oracle.as_bf16_bits(x) for x in xs])
        assert np.array_equal(o16, xcat[:, :n]), rt
        assert np.array_equal(o32, _f32(xcat[:, :n])), rt


def pin_shard_isolation(lib):
    P, m, k, n = 4, 3, 40, 24
    for rt in (False, True):
        xs, y = make_inputs(P, m, k, n, rt, dist="uniform", seed=11)
        for r in range(P):
            iso = [x if i == r else torch.zeros_like(x) for i, x in enumerate(xs)]
            o32, _ = oracle.agmm(iso, y, rt, lib=lib)
            alone, _ = oracle.agmm([xs[r]], y, rt, lib=lib)
            for b in range(P):
                blk = o32[b * m:(b + 1) * m]
                if b == r:
                    assert np.array_equal(blk, alone), (r, rt)
                else:
                    assert np.all(blk == 0.0), (r, b, rt)


def pin_shard_permutation(lib):
    P, m, k, n = 5, 2, 36, 16
    xs, y = make_inputs(P, m, k, n, False, dist="normal", seed=5)
    perm = [3, 0, 4, 1, 2]
    o32, _ = oracle.agmm(xs, y, False, lib=lib)
    p32, _ = oracle.agmm([xs[i] for i in perm], y, False, lib=lib)
    for b, src in enumerate(perm):
        assert np.array_equal(p32[b * m:(b + 1) * m], o32[src * m:(src + 1) * m])


def pin_scale_by_two(lib):
    for rt in (False, True):
        xs, y = make_inputs(2, 6, 64, 24, rt, dist="normal", seed=9)
        o32, o16 = oracle.agmm(xs, y, rt, lib=lib)
        y2 = (y.float() * 2.0).to(torch.bfloat16)  # exact: power-of-two scaling
        t32, t16 = oracle.agmm(xs, y2, rt, lib=lib)
        assert np.array_equal(t32, 2.0 * o32)
        assert np.array_equal(_f32(t16), 2.0 * _f32(o16))


def _bf16_neighbours(v: Fraction):
    """Largest bf16 <= v and smallest bf16 >= v, as (bits, Fraction) pairs."""
    f = float(v)  # correctly rounded to double; then walk in bf16 steps
    b = int(np.array([f], dtype=np.float32).view(np.uint32)[0] >> 16)

    def val(bits):
        return Fraction(float(np.array([bits << 16], dtype=np.uint32).view(np.float32)[0]))

    def step(bits, up):
        # next bf16 toward +inf (up) or -inf
        neg = bits & 0x8000
        mag = bits & 0x7FFF
        if mag == 0:
            return 0x0001 if up else 0x8001
        if (not neg) == up:
            return bits + 1
        return bits - 1

    lo = b
    while val(lo) > v:
        lo = step(lo, False)
    while val(step(lo, True)) <= v:
        lo = step(lo, True)
    hi = lo if val(lo) == v else step(lo, True)
    return (lo, val(lo)), (hi, val(hi))


def _rne_exact(v: Fraction):
    (lb, lv), (hb, hv) = _bf16_neighbours(v)
    if lv == v:
        return lb, None
    dl, dh = v - lv, hv - v
    if dl < dh:
        return lb, (lv + hv) / 2
    if dh < dl:
        return hb, (lv + hv) / 2
    return (lb if (lb & 1) == 0 else hb), (lv + hv) / 2


def pin_bruteforce_exact(lib):
    rng = np.random.default_rng(42)
    for trial in range(6):
        P = int(rng.integers(1, 4))
        m = int(rng.integers(1, 5))
        k = int(rng.integers(1, 33))
        n = int(rng.integers(1, 17))
        rt = bool(trial % 2)
        xs, y = make_inputs(P, m, k, n, rt, dist="uniform", seed=100 + trial)
        o32, o16 = oracle.agmm(xs, y, rt, lib=lib)
        a = [[Fraction(float(v)) for v in row] for row in _cat_f64(xs)]
        b = _ycan_f64(y, rt)
        bf = [[Fraction(float(v)) for v in row] for row in b]
        for i in range(P * m):
            for j in range(n):
                exact = sum((a[i][kk] * bf[kk][j] for kk in range(k)), Fraction(0))
                absum = sum((abs(a[i][kk] * bf[kk][j]) for kk in range(k)), Fraction(0))
                bound = Fraction(gamma(k)) * absum
                assert abs(Fraction(float(o32[i, j])) - exact) <= bound, (trial, i, j)
                if exact == 0:
                    assert float(o32[i, j]) == 0.0
                    continue
                want, mid = _rne_exact(exact)
                if mid is None or abs(exact - mid) > bound:
                    assert int(o16[i, j]) == want, (trial, i, j, hex(int(o16[i, j])), hex(want))


def pin_layout_consistency(lib):
    xs, y_nk = make_inputs(3, 4, 72, 20, True, dist="normal", seed=21)
    a32, a16 = oracle.agmm(xs, y_nk, True, lib=lib)
    b32, b16 = oracle.agmm(xs, y_nk.T.contiguous(), False, lib=lib)
    assert np.array_equal(a32, b32) and np.array_equal(a16, b16)


def pin_double_mode_close(lib):
    xs, y = make_inputs(2, 8, 256, 48, False, dist="normal", seed=13)
    o32, _ = oracle.agmm(xs, y, False, lib=lib)
    o64 = oracle.agmm(xs, y, False, acc="f64", lib=lib)
    a, b = _cat_f64(xs), _ycan_f64(y, False)
    bound = gamma(256) * (np.abs(a) @ np.abs(b))
    assert np.all(np.abs(o32 - o64) <= bound)
    ref = a @ b
    assert np.allclose(o64, ref, rtol=1e-12, atol=1e-12)


def pin_row_range(lib):
    xs, y = make_inputs(4, 5, 96, 32, True, dist="normal", seed=17)
    full32, full16 = oracle.agmm(xs, y, True, lib=lib)
    for (r0, r1) in [(0, 3), (4, 11), (7, 20), (19, 20), (6, 6)]:
        p32, p16 = oracle.agmm(xs, y, True, row_begin=r0, row_end=r1, lib=lib)
        assert np.array_equal(p32, full32[r0:r1]) and np.array_equal(p16, full16[r0:r1])


# ----------------------------------------------------------------------------- fp16 pins
# The fp16 variant changes only the two conversions; these pin them, and the
# product with fp16 operands, against the binary16 layout, PyTorch's casts
# and exact arithmetic.

def _f16_cat_f64(xs):
    # decoded by PyTorch, independently of the oracle
    return np.concatenate([x.float().double().numpy() for x in xs])


def _f16_ycan_f64(y, rt):
    yf = y.float().double().numpy()
    return yf.T if rt else yf


def pin_f16_golden(lib):
    with open(os.path.join(GOLDEN, "f16_rounding.json")) as f:
        g = json.load(f)
    for f32hex, f16hex, why in g["encode"]:
        f = np.array([int(f32hex, 16)], dtype=np.uint32).view(np.float32)
        got = int(oracle.f32_to_f16_bits(f, lib)[0])
        assert got == int(f16hex, 16), (f32hex, hex(got), why)
    for f16hex, f32hex, why in g["decode"]:
        got = oracle.f16_bits_to_f32(np.array([int(f16hex, 16)], dtype=np.uint16), lib).view(np.uint32)[0]
        assert int(got) == int(f32hex, 16), (f16hex, hex(int(got)), why)
    for nan_bits in (0x7FC00000, 0x7F800001, 0xFFC00001):
        f = np.array([nan_bits], dtype=np.uint32).view(np.float32)
        got = int(oracle.f32_to_f16_bits(f, lib)[0])
        assert (got & 0x7C00) == 0x7C00 and (got & 0x03FF) != 0, hex(got)


def pin_f16_vs_torch(lib):
    rng = np.random.default_rng(4321)
    # random signs, fractions and exponents spanning fp16's subnormals to overflow
    nrand = 200_000
    exp = rng.integers(127 - 30, 127 + 18, size=nrand).astype(np.uint32)
    frac = rng.integers(0, 1 << 23, size=nrand).astype(np.uint32)
    sign = rng.integers(0, 2, size=nrand).astype(np.uint32)
    f = ((sign << 31) | (exp << 23) | frac).view(np.float32)
    # exact ties: normal range (discarded 13 bits = 0x1000) and subnormal range
    te = rng.integers(127 - 14, 127 + 16, size=20_000).astype(np.uint32)
    tf = rng.integers(0, 1 << 10, size=20_000).astype(np.uint32)
    ties_n = ((te << 23) | (tf << 13) | 0x1000).view(np.float32)
    ties_s = (rng.integers(0, 1 << 11, size=20_000).astype(np.float32) + 0.5) * np.float32(2.0 ** -24)
    f = np.concatenate([f, ties_n, ties_s, -ties_s])
    ours = oracle.f32_to_f16_bits(f, lib)
    ref = torch.from_numpy(f.copy()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(hex(int(f.view(np.uint32)[i])), hex(int(ours[i])), hex(int(ref[i]))) for i in bad[:5]]
    # every fp16 pattern decodes as PyTorch decodes it
    allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    dec = oracle.f16_bits_to_f32(allb, lib)
    tref = torch.from_numpy(allb.view(np.int16).copy()).view(torch.float16).float().numpy()
    nan = np.isnan(tref)
    assert np.array_equal(np.isnan(dec), nan)
    assert np.array_equal(dec[~nan].view(np.uint32), tref[~nan].view(np.uint32))


def pin_f16_plain_matmul_p1(lib):
    for (m, k, n, rt, dist) in [(7, 64, 24, False, "uniform"), (5, 256, 40, True, "normal"),
                                (33, 130, 17, False, "normal")]:
        xs, y = make_inputs(1, m, k, n, rt, dist=dist, seed=27, dtype="f16")
        o32, _ = oracle.agmm(xs, y, rt, lib=lib)
        a = _f16_cat_f64(xs)
        b = _f16_ycan_f64(y, rt)
        ref = (torch.from_numpy(a) @ torch.from_numpy(b)).numpy()
        bound = gamma(k) * (np.abs(a) @ np.abs(b)) + 1e-30
        err = np.abs(o32.astype(np.float64) - ref)
        assert np.all(err <= bound), (m, k, n, rt, float((err / bound).max()))
        assert np.any(err > 0)


def pin_f16_identity_embedding(lib):
    for rt in (False, True):
        P, m, k, n = 3, 5, 48, 32
        xs, _ = make_inputs(P, m, k, n, rt, dist="normal", seed=33, dtype="f16")
        eye = torch.zeros((k, n), dtype=torch.float32)
        eye[:n, :n] = torch.eye(n)
        y = (eye.T.contiguous() if rt else eye).to(torch.float16)
        o32, o16 = oracle.agmm(xs, y, rt, lib=lib)
        xcat = np.concatenate([oracle.as_bits(x, "f16") for x in xs])
        assert np.array_equal(o16, xcat[:, :n]), rt
        assert np.array_equal(o32, np.concatenate([x.float().numpy() for x in xs])[:, :n]), rt


_F16_TABLE = None


def _f16_finite_table():
    """Every finite fp16 value as an exact Fraction, sorted, with its bits
    (from PyTorch's decoding)."""
    global _F16_TABLE
    if _F16_TABLE is None:
        allb = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
        vals = torch.from_numpy(allb.view(np.int16).copy()).view(torch.float16).double().numpy()
        pairs = {}
        for b, v in zip(allb.tolist(), vals.tolist()):
            if np.isfinite(v) and not (v == 0.0 and b == 0x8000):
                pairs[Fraction(v)] = b
        keys = sorted(pairs)
        _F16_TABLE = (keys, [pairs[q] for q in keys])
    return _F16_TABLE


def _rne_exact_f16(v: Fraction):
    """Round an exact value to fp16, ties to even; returns (bits, midpoint or None)."""
    import bisect

    keys, bits = _f16_finite_table()
    i = bisect.bisect_left(keys, v)
    if i < len(keys) and keys[i] == v:
        return bits[i], None
    lo, hi = i - 1, i
    dl, dh = v - keys[lo], keys[hi] - v
    mid = (keys[lo] + keys[hi]) / 2
    if dl < dh:
        return bits[lo], mid
    if dh < dl:
        return bits[hi], mid
    return (bits[lo] if (bits[lo] & 1) == 0 else bits[hi]), mid


def pin_f16_bruteforce_exact(lib):
    rng = np.random.default_rng(47)
    for trial in range(5):
        P = int(rng.integers(1, 4))
        m = int(rng.integers(1, 5))
        k = int(rng.integers(1, 33))
        n = int(rng.integers(1, 17))
        rt = bool(trial % 2)
        xs, y = make_inputs(P, m, k, n, rt, dist="uniform", seed=200 + trial, dtype="f16")
        o32, o16 = oracle.agmm(xs, y, rt, lib=lib)
        a = [[Fraction(float(v)) for v in row] for row in _f16_cat_f64(xs)]
        bf = [[Fraction(float(v)) for v in row] for row in _f16_ycan_f64(y, rt)]
        for i in range(P * m):
            for j in range(n):
                exact = sum((a[i][kk] * bf[kk][j] for kk in range(k)), Fraction(0))
                absum = sum((abs(a[i][kk] * bf[kk][j]) for kk in range(k)), Fraction(0))
                bound = Fraction(gamma(k)) * absum
                assert abs(Fraction(float(o32[i, j])) - exact) <= bound, (trial, i, j)
                if exact == 0:
                    assert float(o32[i, j]) == 0.0
                    continue
                want, mid = _rne_exact_f16(exact)
                if mid is None or abs(exact - mid) > bound:
                    assert int(o16[i, j]) == want, (trial, i, j, hex(int(o16[i, j])), hex(want))


def pin_bf16_decode_all_patterns(lib):
    # bf16 is the upper half of a binary32 pattern: every one of the 65536
    # patterns decodes, through both of the oracle's decoders, to that
    # binary32 value (compared bit for bit, so NaN payloads count too)
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = (bits.astype(np.uint32) << 16).view(np.float32)
    got = np.empty(65536, dtype=np.float32)
    lib.oracle_bf16_array_to_f32(bits.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)),
                                 got.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), 65536)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    for b in (0x0000, 0x8000, 0x3F80, 0xBF80, 0x7F80, 0xFF80, 0x0001, 0x7FC0):
        assert np.float32(lib.oracle_bf16_to_f32(b)).view(np.uint32) == np.uint32(b) << np.uint32(16)


ALL_PINS = [pin_bf16_golden, pin_bf16_decode_all_patterns, pin_bf16_vs_torch, pin_hand_example, pin_plain_matmul_p1,
            pin_identity_embedding, pin_shard_isolation, pin_shard_permutation, pin_scale_by_two,
            pin_bruteforce_exact, pin_layout_consistency, pin_double_mode_close, pin_row_range,
            pin_f16_golden, pin_f16_vs_torch, pin_f16_plain_matmul_p1, pin_f16_identity_embedding,
            pin_f16_bruteforce_exact]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_thread_count_invariance(oracle_lib):
    xs, y = make_inputs(3, 17, 200, 64, False, dist="normal", seed=2)
    a32, a16 = oracle.agmm(xs, y, False, nthreads=1, lib=oracle_lib)
    b32, b16 = oracle.agmm(xs, y, False, nthreads=4, lib=oracle_lib)
    assert np.array_equal(a32, b32) and np.array_equal(a16, b16)


def test_oracle_rejects_bad_args(oracle_lib):
    xs, y = make_inputs(2, 4, 32, 8, False, dist="normal")
    with pytest.raises(ValueError):
        oracle.agmm(xs, y.T.contiguous()[:, :16], False, lib=oracle_lib)
    with pytest.raises(ValueError):
        oracle.agmm(xs, y, False, row_begin=5, row_end=3, lib=oracle_lib)
    # the C entry point itself rejects a bad range
    import ctypes
    u16p = ctypes.POINTER(ctypes.c_uint16)
    bits = [oracle.as_bf16_bits(x) for x in xs]
    ptrs = (u16p * 2)(*[b.ctypes.data_as(u16p) for b in bits])
    yb = oracle.as_bf16_bits(y)
    out = np.empty((8, 8), dtype=np.float32)
    rc = oracle_lib.oracle_agmm(2, 4, 32, 8, 0, ptrs, yb.ctypes.data_as(u16p), 5, 3, 0,
                                out.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), None, None, 1)
    assert rc == -1


# ----------------------------------------------------------------------------- mutations
# Plausible mistakes planted in copies of oracle.c (on the CPU); each must make
# at least one pin fail.
MUTANTS = {
    "dropped_first_term": ("for (int64_t kk = 0; kk < k; ++kk) {\n                const float a",
                           "for (int64_t kk = 1; kk < k; ++kk) {\n                const float a"),
    "dropped_last_term": ("for (int64_t kk = 0; kk < k; ++kk) {\n                const float a",
                          "for (int64_t kk = 0; kk + 1 < k; ++kk) {\n                const float a"),
    "transposed_operand": ("rhs_transpose ? y[j * k + kk] : y[kk * n + j]",
                           "rhs_transpose ? y[kk * n + j] : y[j * k + kk]"),
    "reversed_rank_order": ("x_shards[g / m_per_device]", "x_shards[(P - 1) - g / m_per_device]"),
    "wrong_sign": ("for (int64_t j = 0; j < n; ++j) acc[j] += a * yr[j];",
                   "for (int64_t j = 0; j < n; ++j) acc[j] -= a * yr[j];"),
    "round_half_up": ("u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0x8000u;"),
    "truncating_cast": ("u += 0x7FFFu + ((u >> 16) & 1u);", "u += 0u;"),
    "wrong_row_in_shard": ("(g % m_per_device) * k", "(g / P % m_per_device) * k"),
    # the fp16 conversions
    "f16_round_half_up": ("(rem > half || (rem == half && (q & 1u)))", "(rem >= half)"),
    "f16_truncating_cast": ("(rem > half || (rem == half && (q & 1u)))", "(0)"),
    "f16_subnormal_scale": ("const int shift = e >= 1 ? 13 : 14 - e;", "const int shift = e >= 1 ? 13 : 13 - e;"),
    "f16_no_overflow": ("if (e >= 31) return (uint16_t)(sign | 0x7C00u);", "if (e >= 32) return (uint16_t)(sign | 0x7C00u);"),
    "f16_decode_bias": ("((uint32_t)(e - 15 + 127) << 23)", "((uint32_t)(e - 16 + 127) << 23)"),
    # the bf16 decoder
    "bf16_decode_shift": ("uint32_t u = ((uint32_t)b) << 16;", "uint32_t u = ((uint32_t)b) << 15;"),
}


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, mutant_dir):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    msrc = os.path.join(mutant_dir, f"{name}.c")
    mlib = os.path.join(mutant_dir, f"lib{name}.so")
    with open(msrc, "w") as f:
        f.write(src.replace(old, new))
    oracle.build(force=True, src=msrc, out=mlib)
    lib = oracle.load(mlib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ArithmeticError):  # a wrong or non-finite result
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
