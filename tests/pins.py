"""Independent references that pin the oracle (test side only).

Nothing here calls the oracle's arithmetic: the tables are enumerated from the
format definitions field by field, rounding is a brute-force nearest search or
an integer carry on the float64 bit pattern, and library conversions (torch,
numpy) serve as the special cases they cover.
"""
import numpy as np


# ---------------------------------------------------------------- tables
def e4m3_table():
    """Values of the 256 E4M3 (fn) codes: sign | exponent(4) | mantissa(3),
    bias 7; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN."""
    vals = np.empty(256, np.float64)
    for code in range(256):
        s = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = s * (m / 8.0) * 2.0 ** -6
        else:
            vals[code] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


def e2m1_table():
    """Values of the 16 E2M1 codes: sign | exponent(2) | mantissa(1), bias 1;
    exponent 0 is subnormal (m/2)."""
    vals = np.empty(16, np.float64)
    for code in range(16):
        s = -1.0 if code & 0x8 else 1.0
        e = (code >> 1) & 0x3
        m = code & 0x1
        vals[code] = s * ((m / 2.0) if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1))
    return vals


# ---------------------------------------------------------------- brute force
def _nearest_code(a, mags, max_code):
    """Codes 0..max_code of the magnitudes `mags` (increasing in code order)
    nearest to each a >= 0; ties go to the even code; a >= the largest
    magnitude gives max_code (satfinite)."""
    a = np.asarray(a, np.float64)
    out = np.empty(a.shape, np.int64)
    flat_a = a.ravel()
    flat_o = out.ravel()
    codes = np.arange(max_code + 1)
    for c0 in range(0, flat_a.size, 1 << 14):
        blk = flat_a[c0:c0 + (1 << 14)]
        d = np.abs(blk[:, None] - mags[None, :max_code + 1])
        dmin = d.min(axis=1, keepdims=True)
        tie = d == dmin
        # among the nearest, prefer an even code, then the smallest
        score = np.where(tie, codes[None, :] % 2 * 1000 + codes[None, :], 10 ** 9)
        res = score.argmin(axis=1)
        res = np.where(blk >= mags[max_code], max_code, res)
        flat_o[c0:c0 + blk.size] = res
    return out


def brute_e4m3(v):
    """RNE + satfinite E4M3 code of each float64 v by nearest search."""
    v = np.asarray(v, np.float64)
    mags = e4m3_table()[:0x7F]  # codes 0x00..0x7E are the finite non-negative values
    mag_code = _nearest_code(np.abs(v), mags, 0x7E)
    sign = np.where(np.signbit(v), 0x80, 0)
    return (mag_code | sign).astype(np.uint8)


def brute_e2m1(v):
    v = np.asarray(v, np.float64)
    mags = e2m1_table()[:8]
    mag_code = _nearest_code(np.abs(v), mags, 7)
    sign = np.where(np.signbit(v), 0x8, 0)
    return (mag_code | sign).astype(np.uint8)


# ---------------------------------------------------------------- dtype rounding
def f64_to_bf16_carry(v):
    """float64 -> bf16 bits by round-half-even integer carry on the float64
    pattern (normal bf16 range only): keep 7 of the 52 fraction bits."""
    v = np.ascontiguousarray(v, np.float64)
    b = v.view(np.uint64)
    drop = np.uint64(45)
    lsb = (b >> drop) & np.uint64(1)
    b = (b + (np.uint64(1) << np.uint64(44)) - np.uint64(1) + lsb) & ~((np.uint64(1) << drop) - np.uint64(1))
    f32 = b.view(np.float64).astype(np.float32)  # exact: 8 significant bits
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(b):
    b = np.ascontiguousarray(b, np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def fp16_bits_to_f64(b):
    return np.ascontiguousarray(b, np.uint16).view(np.float16).astype(np.float64)


def bits_to_f64(b, dt):
    return bf16_bits_to_f64(b) if dt == "bf16" else fp16_bits_to_f64(b)


def f64_to_dt(v, dt):
    if dt == "bf16":
        return f64_to_bf16_carry(v)
    return np.asarray(v, np.float64).astype(np.float16).view(np.uint16)


def ulp(v, dt):
    """Spacing of `dt` at |v| (normal range; subnormal spacing below it)."""
    p, emin = (8, -126) if dt == "bf16" else (11, -14)
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)
    return 2.0 ** (e - (p - 1))


def code_steps(a, b, sign_bit):
    """Ordinal distance between sign-magnitude codes (E4M3: 0x80, E2M1: 0x8);
    +0 and -0 are 0 steps apart."""
    a = np.asarray(a).astype(np.int64)
    b = np.asarray(b).astype(np.int64)
    mask = sign_bit - 1

    def ordinal(c):
        mag = c & mask
        return np.where(c & sign_bit, -mag, mag)

    return np.abs(ordinal(a) - ordinal(b))
