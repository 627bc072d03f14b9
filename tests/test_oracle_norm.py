"""Pins for the oracle's residual add + RMSNorm + FP8 steps.

Closed forms (constant rows, zero rows, power-of-two rows with eps = 0), an
exact residual sum rounded by integer carry, a float64 recompute of the norm,
and the accuracy the pages publish for the fused tail.
"""
import ctypes
import os

import numpy as np
import pytest

import oracle as O
import synth
from tests import pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_kv(name):
    kv = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, *v = line.split()
            kv[k] = v
    return kv


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_residual_is_exact_sum_rounded_once(dt):
    x, r, w = synth.rows_input(11, 64, 512, dt)
    s, _ = O.add_rmsnorm(dt, x, r, w, 1e-6)
    exact = pins.bits_to_f64(x, dt) + pins.bits_to_f64(r, dt)  # exact in float64 here
    assert np.array_equal(s, pins.f64_to_dt(exact, dt))


def test_residual_in_place_alias_is_safe():
    """Writing residual' over the residual buffer gives the same result."""
    x, r, w = synth.rows_input(12, 8, 256, "bf16")
    s_ref, y_ref = O.add_rmsnorm("bf16", x, r, w, 1e-6)
    r2 = r.copy()
    y = np.empty_like(x)
    p16 = lambda a: a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))
    O.lib().oracle_add_rmsnorm(0, p16(x), p16(r2), p16(w), 1e-6, 8, 256, p16(r2), p16(y))
    assert np.array_equal(r2, s_ref) and np.array_equal(y, y_ref)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("c", [0.75, -3.0, 1.0e-2])
def test_constant_row_normalises_to_weight(dt, c):
    """x = c, residual = 0: the mean square is c^2, so y = c / sqrt(c^2 + eps) * w
    (~ sign(c) w when eps << c^2) within one ulp."""
    H = 256
    x = np.tile(pins.f64_to_dt(np.array([c]), dt), (4, H))
    r = np.zeros_like(x)
    _, _, w = synth.rows_input(13, 1, H, dt)
    _, y = O.add_rmsnorm(dt, x, r, w, 1e-6)
    wv = pins.bits_to_f64(w, dt)
    yv = pins.bits_to_f64(y, dt)
    cv = pins.bits_to_f64(x[0, :1], dt)[0]
    ref = cv / np.sqrt(cv * cv + 1e-6) * wv
    assert np.all(np.abs(yv - ref) <= pins.ulp(ref, dt))
    if abs(c) >= 0.5:
        assert np.all(np.abs(yv - np.sign(c) * wv) <= pins.ulp(wv, dt))


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_zero_row_stays_zero(dt):
    H = 128
    x = np.zeros((3, H), np.uint16)
    r = np.zeros_like(x)
    _, _, w = synth.rows_input(14, 1, H, dt)
    s, y, q = O.add_rmsnorm_fp8(dt, x, r, w, 1e-6, 0.05)
    assert np.all(pins.bits_to_f64(s, dt) == 0) and np.all(pins.bits_to_f64(y, dt) == 0)
    assert np.all((q & 0x7F) == 0)
    _, _, packed, sf = O.add_rmsnorm_nvfp4(dt, x, r, w, 1e-6, 448.0)
    assert np.all(sf == 0) and np.all((packed & 0x77) == 0)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("H", [16, 48, 1024, 7168])
def test_power_of_two_rows_with_zero_eps_give_exact_weight(dt, H):
    """Rows of +-2^k with eps = 0: mean square 4^k, sqrt 2^k, rstd 2^-k are all
    exact, so y = +-w bit for bit."""
    rng = np.random.default_rng(H)
    rows = 6
    k = rng.integers(-6, 6, rows)
    sign = rng.choice([-1.0, 1.0], (rows, H))
    xv = sign * (2.0 ** k)[:, None]
    x = pins.f64_to_dt(xv, dt)
    r = np.zeros_like(x)
    _, _, w = synth.rows_input(15, 1, H, dt)
    _, y = O.add_rmsnorm(dt, x, r, w, 0.0)
    expect = np.where(sign < 0, w ^ np.uint16(0x8000), w)
    assert np.array_equal(y, expect)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("H", [128, 1024, 7168])
def test_norm_within_one_ulp_of_float64_recompute(dt, H):
    x, r, w = synth.rows_input(16, 32, H, dt, res_std=2.0)
    s, y = O.add_rmsnorm(dt, x, r, w, 1e-6)
    sv = pins.bits_to_f64(s, dt)
    rstd = 1.0 / np.sqrt(np.mean(sv * sv, axis=1, keepdims=True) + 1e-6)
    y64 = sv * rstd * pins.bits_to_f64(w, dt)[None, :]
    err = np.abs(pins.bits_to_f64(y, dt) - y64)
    assert np.all(err <= pins.ulp(y64, dt))


def test_published_accuracy_of_fused_tail():
    """The pages report residual max error 0 and RMSNorm max error 0.00390 for
    the FP16 fused tail (one fp16 ulp for |y| in [4, 8)); the oracle stays
    within both against an exact / float64 recompute, on the pages' [64, 8192]
    FP16 tail shape."""
    kv = _read_kv("published_accuracy.txt")
    assert kv["dtype"] == ["fp16"]
    res_tol = float(kv["residual_max_abs_err"][0])
    norm_tol = float(kv["rmsnorm_max_abs_err"][0])
    x, r, w = synth.rows_input(0, 64, 8192, "fp16")
    s, y = O.add_rmsnorm("fp16", x, r, w, 1e-6)
    sv = pins.fp16_bits_to_f64(s)
    exact = pins.fp16_bits_to_f64(x) + pins.fp16_bits_to_f64(r)
    assert np.max(np.abs(sv - exact.astype(np.float16).astype(np.float64))) <= res_tol
    rstd = 1.0 / np.sqrt(np.mean(sv * sv, axis=1, keepdims=True) + 1e-6)
    y64 = sv * rstd * pins.fp16_bits_to_f64(w)[None, :]
    in_range = np.abs(y64) < 8.0
    err = np.abs(pins.fp16_bits_to_f64(y) - y64)[in_range]
    # 0.00390 is 2^-8 printed to three significant figures
    assert err.max() <= max(norm_tol, 2.0 ** -8)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("scale", [0.05, 0.0137])
def test_fp8_codes_are_nearest_e4m3_of_quotient(dt, scale):
    x, r, w = synth.rows_input(17, 16, 1024, dt, res_std=2.0)
    s, y, q = O.add_rmsnorm_fp8(dt, x, r, w, 1e-6, scale)
    v = (pins.bits_to_f64(y, dt).astype(np.float32) / np.float32(scale)).astype(np.float64)
    assert np.array_equal(q, pins.brute_e4m3(v))
    # and the dequantised value is within half an E4M3 spacing of y
    deq = pins.e4m3_table()[q] * scale
    yv = pins.bits_to_f64(y, dt)
    unsat = np.abs(v) < 448
    sp = np.where(np.abs(v) < 2.0 ** -6, 2.0 ** -9,
                  2.0 ** (np.floor(np.log2(np.maximum(np.abs(v), 1e-30))) - 3))
    assert np.all(np.abs(deq - yv)[unsat] <= (sp * scale * 0.5 * (1 + 1e-6))[unsat])


def test_fp8_worked_value():
    """y = 1 with the dequant scale 0.05: 1/0.05 rounds to 20 in fp32, which is
    exactly representable in E4M3 (1.25 * 2^4: exponent field 11, mantissa 2)."""
    y = np.array([0x3F80, 0xBF80], np.uint16)  # bf16 +1, -1
    q = O.quant_fp8("bf16", y, 0.05)
    assert list(q) == [0x5A, 0xDA]


def test_amax_and_scales():
    x, r, w = synth.rows_input(18, 8, 256, "bf16")
    _, y = O.add_rmsnorm("bf16", x, r, w, 1e-6)
    a = O.amax("bf16", y)
    assert a == np.max(np.abs(pins.bf16_bits_to_f64(y)))
    assert O.fp8_scale_from_amax(a) == float(np.float32(a) / np.float32(448.0))
    assert O.nvfp4_gs_from_amax(a) == float(np.float32(2688.0) / np.float32(a))


# ------------------------------------------------------------- dynamic scales
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_per_row_scales_are_row_amax_over_448(dt):
    """Per-token FP8: each row's scale is amax(|y_row|)/448 in fp32, the row's
    largest magnitude maps to code 0x7E (448) and every code is the nearest
    E4M3 of y/scale; an all-zero row gets scale 1 and zero codes."""
    x, r, w = synth.rows_input(21, 40, 512, dt, res_std=2.0)
    x[3] = 0
    r[3] = 0
    _, y = O.add_rmsnorm(dt, x, r, w, 1e-6)
    q, sc = O.quant_fp8_per_row(dt, y)
    yv = pins.bits_to_f64(y, dt)
    amax = np.abs(yv).max(axis=1).astype(np.float32)
    expect = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    assert np.array_equal(sc, expect)
    assert sc[3] == 1.0 and np.all((q[3] & 0x7F) == 0)
    v = (yv.astype(np.float32) / sc[:, None]).astype(np.float64)
    assert np.array_equal(q, pins.brute_e4m3(v))
    nz = amax > 0
    assert np.all(np.max(q[nz] & 0x7F, axis=1) == 0x7E)


def test_dynamic_tensor_scales():
    assert O.fp8_dynamic_scale(0.0) == 1.0 and O.nvfp4_dynamic_gs(0.0) == 1.0
    assert O.fp8_dynamic_scale(4.48) == float(np.float32(4.48) / np.float32(448.0))
    assert O.nvfp4_dynamic_gs(6.0) == 448.0
