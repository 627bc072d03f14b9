"""Pins for the order of the fp32 roundings the oracle states.

The pages fix the operations but not how each fp32 step is rounded, so the
oracle states one order (true IEEE division by the FP8 scale, block scale
E4M3(f32(f32(gs * amax) / 6)), factor f32(gs / scale)).  A natural
alternative (multiplying by a rounded reciprocal) usually gives the same codes,
so these tests search, in numpy float32, for inputs where the two orders fall
on different sides of a rounding tie of the target format, and check that the
oracle takes the stated order.
"""
import numpy as np

import oracle as O
from tests import pins

f32 = np.float32


def _scan(center, n):
    """n consecutive float32 values around `center`."""
    c = np.float32(center).view(np.int32)
    return (c + np.arange(-n // 2, n // 2, dtype=np.int32)).view(np.float32)


def _bf16(bits):
    return f32((np.uint32(bits) << np.uint32(16)).view(np.float32))


def _e4m3_up_ties():
    """E4M3 midpoints whose tie resolves upward (the upper neighbour has the
    even code): 1.1875, 1.4375, 1.6875, 1.9375 times powers of two."""
    return [f32(m * 2.0 ** k) for k in range(-2, 3) for m in (1.1875, 1.4375, 1.6875, 1.9375)]


def test_fp8_divides_by_the_scale():
    found = None
    for yb in range(0x3F80, 0x4080):  # bf16 values in [1, 4)
        y = _bf16(yb)
        for m in _e4m3_up_ties():
            s = _scan(y / m, 64)
            q_div = y / s
            q_rcp = y * (f32(1.0) / s)
            hit = (q_div == m) & (q_rcp < m)
            if hit.any():
                found = (yb, float(s[hit][0]), float(m), float(q_rcp[hit][0]))
                break
        if found:
            break
    assert found is not None
    yb, scale, m, q_alt = found
    code = O.quant_fp8("bf16", np.array([yb], np.uint16), scale)[0]
    assert pins.e4m3_table()[code] > m  # the tie, resolved to the even (upper) code
    assert pins.brute_e4m3(np.array([q_alt]))[0] != code


def test_block_scale_divides_by_six():
    found = None
    for ab in range(0x4080, 0x4100):  # bf16 amax values in [4, 8)
        a = _bf16(ab)
        for m in _e4m3_up_ties():
            gs = _scan(f32(6.0) * m / a, 64)
            t1 = gs * a
            t_div = t1 / f32(6.0)
            t_rcp = t1 * (f32(1.0) / f32(6.0))
            # t1 * f32(1/6) is never below t1 / 6 (f32(1/6) > 1/6), so the
            # two orders can only part where the quotient is just under a tie
            hit = (t_div < m) & (t_rcp >= m)
            if hit.any():
                found = (ab, float(gs[hit][0]), float(m), float(t_rcp[hit][0]))
                break
        if found:
            break
    assert found is not None
    ab, g, m, t_alt = found
    y = np.zeros((1, 16), np.uint16)
    y[0, 0] = ab
    _, sf = O.quant_nvfp4("bf16", y, g)
    assert pins.e4m3_table()[sf[0, 0]] < m  # the quotient is below the tie
    assert pins.brute_e4m3(np.array([t_alt]))[0] != sf[0, 0]


def test_encode_factor_is_gs_over_scale():
    """With amax 6 and gs in (1.0625, 1.1875) the block scale is 1.125 and the
    factor f32(gs / 1.125).  Search a gs and a bf16 y in [2, 6) for which
    y * factor and y * (1 / f32(1.125 / gs)) round to different E2M1 codes."""
    sfv = f32(1.125)
    gs = _scan(sfv, 1 << 20)
    gs = gs[(gs > f32(1.0625)) & (gs < f32(1.1875))]
    enc1 = gs / sfv
    enc2 = f32(1.0) / (sfv / gs)
    part = enc1 != enc2
    gs, enc1, enc2 = gs[part], enc1[part], enc2[part]
    found = None
    for yb in range(0x4000, 0x40C0):
        yv = _bf16(yb)
        v1 = (yv * enc1).astype(np.float64)
        v2 = (yv * enc2).astype(np.float64)
        near = np.abs(v1 - np.round(v1 * 2) / 2) < 1e-3  # only values near a tie can part
        if not near.any():
            continue
        c1, c2 = pins.brute_e2m1(v1[near]), pins.brute_e2m1(v2[near])
        hit = c1 != c2
        if hit.any():
            found = (yb, float(gs[near][hit][0]), int(c1[hit][0]), int(c2[hit][0]))
            break
    assert found is not None
    yb, g, c_stated, c_alt = found
    y = np.zeros((1, 16), np.uint16)
    y[0, 0] = 0x40C0  # amax 6 sets the block scale
    y[0, 1] = yb
    packed, sf = O.quant_nvfp4("bf16", y, g)
    assert pins.e4m3_table()[sf[0, 0]] == 1.125
    assert packed[0, 0] >> 4 == c_stated != c_alt
