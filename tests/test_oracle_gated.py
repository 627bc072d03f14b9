"""Pins of the oracle's gated RMSNorm (the fused gated RMSNorm + NVFP4 op of
"Add AutoDeploy NVFP4 RMSNorm quant fusion", Changes).  The page gives no
formula; the reading is g = dt(x * dt(silu(z))), silu(z) = z / (1 + e^-z),
then the RMSNorm and NVFP4 steps of the plain path on g.

- silu against torch's float64 SiLU (a library routine) over every finite
  bf16 and fp16 value, rounded to fp32 and then to the dtype;
- closed forms: silu(0) = 0, silu(z) = z where e^-z is below half an fp32
  ulp, silu(z) = -0 where e^-z overflows;
- the gate reduces to the plain path: with z = 32 (silu(32) rounds to 32)
  and eps = 0, g = 32 x exactly and the norm output equals the plain
  residual-add path's on x with a residual of -0 (x + (-0) = x, signed zeros
  included), bit for bit, because every step commutes with a power-of-two
  scaling;
- an all-zero gate gives zero rows: signed zero codes and zero block scales.
"""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from tests import pins


def _all_finite(dt):
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = pins.bits_to_f64(b, dt)
    return b[np.isfinite(v)]


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_silu_matches_torch_float64_silu_on_every_value(dt):
    z = _all_finite(dt)
    z64 = torch.from_numpy(pins.bits_to_f64(z, dt))
    ref = torch.nn.functional.silu(z64).numpy()
    ref_bits = synth.to_bits(ref.astype(np.float32).astype(np.float64), dt)
    got = O.silu_dt(dt, z)
    bad = got != ref_bits
    assert not bad.any(), "silu differs at %d values, first z bits 0x%04x" % (
        int(bad.sum()), int(z[bad][0]))


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_silu_closed_forms(dt):
    enc = lambda v: int(synth.to_bits(np.array([v]), dt)[0])
    assert O.silu_dt(dt, np.array([enc(0.0)], np.uint16))[0] == enc(0.0)
    # e^-z below half an ulp of 1 in fp32 (z >= 17): silu(z) = z
    for v in (17.0, 32.0, 1000.0):
        assert O.silu_dt(dt, np.array([enc(v)], np.uint16))[0] == enc(v)
    # e^-z overflows double for -z > 710 (bf16 only reaches that): -0
    if dt == "bf16":
        assert O.silu_dt(dt, np.array([enc(-1000.0)], np.uint16))[0] == 0x8000
    # odd-part identity silu(z) - silu(-z) = z, within the two roundings
    z = synth.to_bits(np.linspace(-8, 8, 161), dt)
    zn = synth.to_bits(-pins.bits_to_f64(z, dt), dt)
    a = pins.bits_to_f64(O.silu_dt(dt, z), dt)
    b = pins.bits_to_f64(O.silu_dt(dt, zn), dt)
    zv = pins.bits_to_f64(z, dt)
    assert np.all(np.abs(a - b - zv) <= pins.ulp(a, dt) + pins.ulp(b, dt))


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_gate_of_32_reduces_to_the_plain_path(dt):
    rows, hidden = 24, 1040
    x, _, w = synth.rows_input(3, rows, hidden, dt)
    z = np.full((rows, hidden), synth.to_bits(np.array([32.0]), dt)[0], np.uint16)
    zeros = np.full_like(x, 0x8000)  # -0: x + (-0) = x, signed zeros included
    x[0, :8] = [0x0000, 0x8000] * 4  # signed zeros in x keep their sign on both paths
    g, y = O.gated_rmsnorm(dt, x, z, w, 0.0)
    s_ref, y_ref = O.add_rmsnorm(dt, x, zeros, w, 0.0)
    assert np.array_equal(pins.bits_to_f64(g, dt), 32.0 * pins.bits_to_f64(x, dt))
    assert np.array_equal(y, y_ref)
    gs = 100.0
    _, _, p, sf = O.gated_rmsnorm_nvfp4(dt, x, z, w, 0.0, gs)
    p_ref, sf_ref = O.quant_nvfp4(dt, y_ref, gs)
    assert np.array_equal(p, p_ref) and np.array_equal(sf, sf_ref)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_zero_gate_gives_zero_rows(dt):
    rows, hidden = 4, 64
    x, _, w = synth.rows_input(4, rows, hidden, dt)
    z = np.zeros((rows, hidden), np.uint16)
    g, y, p, sf = O.gated_rmsnorm_nvfp4(dt, x, z, w, 1e-6, 50.0)
    assert np.all(pins.bits_to_f64(g, dt) == 0.0) and np.all(pins.bits_to_f64(y, dt) == 0.0)
    assert np.all(sf == 0) and np.all((p & 0x77) == 0)  # magnitude bits of both nibbles


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_gate_product_is_the_exact_product_rounded_once(dt):
    # x and dt(silu(z)) have at most 11 significant bits each, so their fp32
    # product is exact: g is the exact product rounded once to the dtype
    rows, hidden = 16, 512
    x, z, w = synth.rows_input(5, rows, hidden, dt, res_std=3.0)
    g, _ = O.gated_rmsnorm(dt, x, z, w, 1e-6)
    exact = pins.bits_to_f64(x, dt) * pins.bits_to_f64(O.silu_dt(dt, z), dt)
    assert np.array_equal(g, synth.to_bits(exact, dt))
    # and the gate is not the unrounded fp32 silu: that reading differs here
    s32 = (pins.bits_to_f64(z, dt) / (1.0 + np.exp(-pins.bits_to_f64(z, dt)))).astype(np.float32)
    other = synth.to_bits((pins.bits_to_f64(x, dt).astype(np.float32) * s32).astype(np.float64), dt)
    assert not np.array_equal(g, other)
