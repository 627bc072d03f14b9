"""Pins for the oracle's number formats (bf16, fp16, E4M3, E2M1).

The oracle rounds with a frexp / nearbyint construction; these tests check it
against brute-force nearest searches over tables enumerated field by field,
against integer-carry rounding, and against torch / numpy conversions where
those libraries implement the same format.
"""
import numpy as np
import pytest
import torch

import oracle as O
from tests import pins


def _all_finite(dt):
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = pins.bits_to_f64(b, dt)
    ok = np.isfinite(v)
    return b[ok], v[ok]


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_dtype_decode_and_roundtrip_exhaustive(dt):
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = pins.bits_to_f64(b, dt)
    got = O.dt_to_double(dt, b)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # every non-NaN pattern survives decode -> encode
    back = O.dt_from_double(dt, got[~nan])
    assert np.array_equal(back, b[~nan])


def _rounding_probe_values(rng, dt):
    """float32 values around every rounding decision of `dt`: random values
    over the whole exponent range, exact ties (half an ulp above a dtype
    value), one float32 ulp either side of the ties, overflow and subnormals."""
    b, v = _all_finite(dt)
    v = v[v != 0]
    vals = [rng.standard_normal(20000) * 10.0 ** rng.uniform(-8, 8, 20000)]
    u = pins.ulp(v, dt)
    mid = (v + np.sign(v) * u / 2.0).astype(np.float32).astype(np.float64)
    f32_next_up = np.nextafter(mid.astype(np.float32), np.float32(np.inf)).astype(np.float64)
    f32_next_dn = np.nextafter(mid.astype(np.float32), np.float32(-np.inf)).astype(np.float64)
    vals += [mid, f32_next_up, f32_next_dn]
    big = 3.3e38 if dt == "bf16" else 65519.0
    vals.append(np.array([big, -big, 65520.0, 65504.0, 1e-45, -1e-45, 6e-8, 3e-8, 0.0, -0.0]))
    out = np.concatenate(vals).astype(np.float32)
    return out[np.isfinite(out)].astype(np.float64)


def test_bf16_encoder_matches_torch():
    rng = np.random.default_rng(1)
    v = _rounding_probe_values(rng, "bf16")
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.dt_from_double("bf16", v)
    assert np.array_equal(got, ref)


def test_fp16_encoder_matches_numpy():
    rng = np.random.default_rng(2)
    v = _rounding_probe_values(rng, "fp16")
    ref = v.astype(np.float32).astype(np.float16).view(np.uint16)
    got = O.dt_from_double("fp16", v)
    assert np.array_equal(got, ref)


def test_bf16_encoder_matches_integer_carry():
    rng = np.random.default_rng(3)
    # normal-range float64 values, including exact float64 ties
    v = rng.standard_normal(200000) * 2.0 ** rng.integers(-60, 60, 200000)
    b, base = _all_finite("bf16")
    base = base[(np.abs(base) > 1e-30) & (np.abs(base) < 1e30)]
    ties = base + np.sign(base) * pins.ulp(base, "bf16") / 2.0
    v = np.concatenate([v, ties])
    assert np.array_equal(O.dt_from_double("bf16", v), pins.f64_to_bf16_carry(v))


def test_e4m3_decode_table():
    tab = pins.e4m3_table()
    got = O.e4m3_to_double(np.arange(256, dtype=np.uint8))
    nan = np.isnan(tab)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    assert np.array_equal(got[~nan], tab[~nan])
    # values the OCP format states: max 448, min subnormal 2^-9,
    # min normal 2^-6, one
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9
    assert got[0x08] == 2.0 ** -6 and got[0x38] == 1.0
    # and torch's float8_e4m3fn agrees on every code
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(t), nan) and np.array_equal(t[~nan], tab[~nan])


def test_e2m1_decode_table():
    got = O.e2m1_to_double(np.arange(16, dtype=np.uint8))
    assert np.array_equal(got, pins.e2m1_table())
    assert list(got[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("scale", [1.0, 0.05, 0.0123456])
def test_e4m3_encoder_exhaustive_vs_brute_force(dt, scale):
    """Every finite dtype value y, divided by the scale in fp32, encodes to
    the nearest E4M3 code (ties to even, satfinite)."""
    _, y = _all_finite(dt)
    v = (y.astype(np.float32) / np.float32(scale)).astype(np.float64)
    got = O.e4m3_from_double(v)
    ref = pins.brute_e4m3(v)
    assert np.array_equal(got, ref)


def test_e4m3_encoder_matches_torch_in_range():
    """torch's float8_e4m3fn cast is RNE but overflows to NaN instead of
    saturating, so it covers |v| <= 448 only."""
    rng = np.random.default_rng(4)
    tab = pins.e4m3_table()[:0x7F]
    mids = (tab[:-1] + tab[1:]) / 2.0
    v = np.concatenate([rng.uniform(-448, 448, 100000),
                        rng.standard_normal(100000) * 2.0 ** rng.integers(-14, 8, 100000),
                        mids, -mids, np.nextafter(mids, 0), np.nextafter(mids, 1e9)])
    v = v[np.abs(v) <= 448].astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_from_double(v.astype(np.float64))
    assert np.array_equal(got, ref)


def test_e4m3_special_cases():
    f = lambda x: int(O.e4m3_from_double(np.array([x]))[0])
    assert f(448.0) == 0x7E and f(1e9) == 0x7E and f(-np.inf) == 0xFE
    assert f(464.0) == 0x7E  # tie between 448 and the (NaN) next code saturates
    assert f(-0.0) == 0x80 and f(0.0) == 0x00
    assert f(2.0 ** -10) == 0x00  # tie between 0 and 2^-9: even code 0
    assert f(3 * 2.0 ** -10) == 0x02  # tie between 2^-9 and 2^-8: even code 2
    assert f(np.nan) == 0x7F


def test_e2m1_encoder_brute_force_and_ties():
    tab = pins.e2m1_table()[:8]
    mids = (tab[:-1] + tab[1:]) / 2.0
    dense = np.linspace(-8, 8, 16001)
    around = np.concatenate([mids, np.nextafter(mids, 0), np.nextafter(mids, 10)])
    v = np.concatenate([dense, around, -around, [6.0, 6.5, 100.0, -100.0, 0.0, -0.0]])
    got = O.e2m1_from_double(v)
    assert np.array_equal(got, pins.brute_e2m1(v))
    # the tie points, written out: 0.25->0, 0.75->1, 1.25->1, 1.75->2,
    # 2.5->2, 3.5->4, 5->4
    t = O.e2m1_to_double(O.e2m1_from_double(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])))
    assert list(t) == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    assert int(O.e2m1_from_double(np.array([-0.0]))[0]) == 0x8
