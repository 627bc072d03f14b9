"""Pins for the oracle's NVFP4 quantiser: hand-worked blocks, exact round
trips, brute-force code search and the dequantisation error bound."""
import os

import numpy as np
import pytest

import oracle as O
import synth
from tests import pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _worked_blocks():
    blocks, cur = [], None
    with open(os.path.join(GOLDEN, "nvfp4_worked_blocks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "block":
                cur = {"name": vals[0]}
                blocks.append(cur)
            elif key == "gs":
                cur["gs"] = float(vals[0])
            elif key == "y":
                cur["y"] = np.array([float(v) for v in vals])
            elif key == "sf":
                cur["sf"] = int(vals[0], 16)
            elif key == "packed":
                cur["packed"] = np.array([int(v, 16) for v in vals], np.uint8)
    return blocks


@pytest.mark.parametrize("blk", _worked_blocks(), ids=lambda b: b["name"])
def test_hand_worked_blocks(blk):
    y = pins.f64_to_bf16_carry(blk["y"]).reshape(1, 16)
    assert np.array_equal(pins.bf16_bits_to_f64(y)[0], blk["y"])  # exact in bf16
    packed, sf = O.quant_nvfp4("bf16", y, blk["gs"])
    assert sf[0, 0] == blk["sf"]
    assert np.array_equal(packed[0], blk["packed"])


@pytest.mark.parametrize("k", [-6, -1, 0, 3, 8])
def test_exactly_representable_rows_round_trip(k):
    """eps = 0 and rows of +-1 give y = +-w exactly.  With weights drawn from
    the E2M1 magnitudes times 2^k, a block amax of 6*2^k and gs = 1, the block
    scale is exactly 2^k, the factor 2^-k, every y*factor is an E2M1 value and
    the dequantised tensor equals y bit for bit."""
    H, rows = 256, 4
    rng = np.random.default_rng(100 + k)
    mags = np.array([0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    wv = rng.choice(mags, H)
    wv[::16] = 6.0  # every block reaches amax 6 * 2^k
    wv = wv * 2.0 ** k
    w = pins.f64_to_bf16_carry(wv)
    sign = rng.choice([-1.0, 1.0], (rows, H))
    x = pins.f64_to_bf16_carry(sign)
    r = np.zeros_like(x)
    _, y, packed, sf = O.add_rmsnorm_nvfp4("bf16", x, r, w, 0.0, 1.0)
    assert np.array_equal(pins.bf16_bits_to_f64(y), sign * wv[None, :])
    assert np.all(pins.e4m3_table()[sf] == 2.0 ** k)
    deq = O.nvfp4_dequant(packed, sf, 1.0)
    assert np.array_equal(deq, sign * wv[None, :])
    # codes in closed form: index of |w| / 2^k among the E2M1 magnitudes
    idx = np.searchsorted(pins.e2m1_table()[:8], wv / 2.0 ** k)
    codes = np.where(sign < 0, 8, 0) | idx[None, :]
    assert np.array_equal(packed, (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8))


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("H", [16, 128, 7168])
def test_codes_and_scales_by_brute_force(dt, H):
    """Each block scale is the nearest E4M3 code of gs*amax/6 and each code the
    nearest E2M1 of y times gs/scale (with the fp32 roundings of the steps)."""
    x, r, w = synth.rows_input(19, 24, H, dt, outlier_frac=0.01)
    _, y = O.add_rmsnorm(dt, x, r, w, 1e-6)
    gs = O.nvfp4_gs_from_amax(O.amax(dt, y))
    packed, sf = O.quant_nvfp4(dt, y, gs)
    yv = pins.bits_to_f64(y, dt).reshape(24, H // 16, 16)
    a = np.abs(yv).max(axis=2).astype(np.float32)
    t2 = (np.float32(gs) * a) / np.float32(6.0)
    assert np.array_equal(sf, pins.brute_e4m3(t2.astype(np.float64)))
    sfv = pins.e4m3_table()[sf].astype(np.float32)
    with np.errstate(divide="ignore"):
        enc = np.where(sfv == 0, np.float32(0), np.float32(gs) / sfv).astype(np.float32)
    v = (yv.astype(np.float32) * enc[:, :, None]).astype(np.float64).reshape(24, H)
    codes = pins.brute_e2m1(v)
    assert np.array_equal(packed, (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8))


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_dequant_error_within_one_block_step(dt):
    """With a normal block scale, every dequantised value is within one block
    quantisation step (half the top E2M1 spacing 2, times scale/gs) of y;
    scales never exceed 448."""
    x, r, w = synth.rows_input(20, 64, 2048, dt, outlier_frac=0.01)
    _, y = O.add_rmsnorm(dt, x, r, w, 1e-6)
    gs = O.nvfp4_gs_from_amax(O.amax(dt, y))
    packed, sf = O.quant_nvfp4(dt, y, gs)
    sfv = pins.e4m3_table()[sf]
    assert np.all(sfv <= 448.0)
    deq = O.nvfp4_dequant(packed, sf, gs)
    yv = pins.bits_to_f64(y, dt)
    step = np.repeat(sfv / gs, 16, axis=1)
    normal = np.repeat(sfv >= 2.0 ** -6, 16, axis=1)
    assert np.all(np.abs(deq - yv)[normal] <= step[normal] * (1 + 1e-6))


def test_all_zero_block():
    y = np.zeros((2, 32), np.uint16)
    y[1, 16:] = 0x3F80  # second block of row 1 is all ones
    packed, sf = O.quant_nvfp4("bf16", y, 448.0)
    assert list(sf[0]) == [0, 0] and sf[1, 0] == 0 and sf[1, 1] != 0
    assert np.all(packed[0] == 0) and np.all(packed[1, :8] == 0)
