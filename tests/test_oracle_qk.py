"""Pins for the oracle's per-head Q/K RMSNorm + NeoX RoPE + FP8 store."""
import numpy as np
import pytest

import oracle as O
import synth
from tests import pins

D = 128


def _setup(dt="bf16", T=32, H=4, seed=21):
    q, k, qw, kw, pos, cs = synth.qk_input(seed, T, H, 2, D, dt)
    return q, qw, pos, cs


def test_rope_table_closed_form():
    cs = synth.rope_cos_sin(64, D, 1.0e6)
    p = np.arange(64)
    # frequency 0 is 1 rad per position; position 0 is the identity rotation
    assert np.array_equal(cs[:, 0], np.cos(p).astype(np.float32))
    assert np.array_equal(cs[:, 64], np.sin(p).astype(np.float32))
    assert np.all(cs[0, :64] == 1.0) and np.all(cs[0, 64:] == 0.0)
    # frequency 32 is theta^(-1/2) = 1e-3
    assert np.allclose(cs[:, 32], np.cos(p * 1e-3), rtol=0, atol=1e-7)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_position_zero_is_norm_only(dt):
    """At position 0 the rotation is the identity, so the Q/K output equals the
    per-head RMSNorm of the plain add + RMSNorm oracle (zero residual)."""
    q, qw, pos, cs = _setup(dt)
    T, H = q.shape[:2]
    zero_pos = np.zeros(T, np.int32)
    o = O.qk_rmsnorm_rope(dt, q.reshape(-1), H * D, T, H, D, qw, 1e-6, zero_pos, cs)
    _, n = O.add_rmsnorm(dt, q.reshape(T * H, D), np.zeros((T * H, D), np.uint16), qw, 1e-6)
    assert np.array_equal(o.reshape(T * H, D), n)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_rotation_within_rounding_of_float64(dt):
    """o_lo = n_lo cos - n_hi sin, o_hi = n_hi cos + n_lo sin (NeoX halves),
    recomputed in float64 from the rounded norm."""
    q, qw, pos, cs = _setup(dt, T=64)
    T, H = q.shape[:2]
    o = O.qk_rmsnorm_rope(dt, q.reshape(-1), H * D, T, H, D, qw, 1e-6, pos, cs)
    _, n = O.add_rmsnorm(dt, q.reshape(T * H, D), np.zeros((T * H, D), np.uint16), qw, 1e-6)
    nv = pins.bits_to_f64(n, dt).reshape(T, H, D)
    c = cs[pos][:, None, :64].astype(np.float64)
    s = cs[pos][:, None, 64:].astype(np.float64)
    lo, hi = nv[..., :64], nv[..., 64:]
    ref = np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)
    ov = pins.bits_to_f64(o, dt)
    # the dtype rounding (<= 1/2 ulp) plus the fp32 roundings of the two
    # products and the sum (each <= 2^-24 relative to its operand)
    mag = np.concatenate([np.abs(lo * c) + np.abs(hi * s), np.abs(hi * c) + np.abs(lo * s)], axis=-1)
    tol = 0.5 * pins.ulp(ref, dt) + 2.0 ** -22 * mag
    assert np.all(np.abs(ov - ref) <= tol)


def test_rotation_preserves_pair_norm():
    q, qw, pos, cs = _setup("bf16", T=128)
    T, H = q.shape[:2]
    o = O.qk_rmsnorm_rope("bf16", q.reshape(-1), H * D, T, H, D, qw, 1e-6, pos, cs)
    _, n = O.add_rmsnorm("bf16", q.reshape(T * H, D), np.zeros((T * H, D), np.uint16), qw, 1e-6)
    nv = pins.bf16_bits_to_f64(n).reshape(T, H, D)
    ov = pins.bf16_bits_to_f64(o)
    rn = np.hypot(nv[..., :64], nv[..., 64:])
    ro = np.hypot(ov[..., :64], ov[..., 64:])
    # each output is within half a bf16 ulp (relative 2^-8) of the exact rotation
    assert np.all(np.abs(ro - rn) <= 2.0 ** -7 * rn + 1e-30)


def test_token_stride_reads_a_fused_buffer():
    """Q taken out of a [T, Hq + Hk + Hv, D] fused buffer by token stride gives
    the same result as a contiguous Q."""
    q, qw, pos, cs = _setup("bf16", T=16, H=4)
    T, H = q.shape[:2]
    fused = np.zeros((T, 8, D), np.uint16)
    fused[:, :H] = q
    o1 = O.qk_rmsnorm_rope("bf16", q.reshape(-1), H * D, T, H, D, qw, 1e-6, pos, cs)
    o2 = O.qk_rmsnorm_rope("bf16", fused.reshape(-1), 8 * D, T, H, D, qw, 1e-6, pos, cs)
    assert np.array_equal(o1, o2)


def test_fp8_store_is_quantiser_of_rotated_values():
    q, qw, pos, cs = _setup("bf16")
    T, H = q.shape[:2]
    o, qq = O.qk_rmsnorm_rope_fp8("bf16", q.reshape(-1), H * D, T, H, D, qw, 1e-6, pos, cs, 0.01)
    assert np.array_equal(qq, O.quant_fp8("bf16", o, 0.01))
    v = (pins.bf16_bits_to_f64(o).astype(np.float32) / np.float32(0.01)).astype(np.float64)
    assert np.array_equal(qq, pins.brute_e4m3(v))


def test_out_of_range_positions_are_clamped():
    q, qw, pos, cs = _setup("bf16", T=8)
    T, H = q.shape[:2]
    bad = np.array([-5, 0, 1, 2, 100, 7, 8, 9], np.int32)
    clamped = np.clip(bad, 0, 7).astype(np.int32)
    o1 = O.qk_rmsnorm_rope("bf16", q.reshape(-1), H * D, T, H, D, qw, 1e-6, bad, cs[:8])
    o2 = O.qk_rmsnorm_rope("bf16", q.reshape(-1), H * D, T, H, D, qw, 1e-6, clamped, cs[:8])
    assert np.array_equal(o1, o2)


# ---------------------------------------------------------------- partial rotary
# The FP8-nope + dtype-rope KV pool: RMSNorm over the whole head, NeoX RoPE
# over its last rope_dim elements only (reading of the pool's head split).
def _partial(dt, q, qw, rope_dim, pos, T=None):
    T, H = q.shape[:2]
    cs = synth.rope_cos_sin(max(int(pos.max()) + 1, 1), rope_dim, 1.0e6)
    o = O.qk_rmsnorm_rope_partial(dt, q.reshape(-1), H * D, T, H, D, rope_dim, qw, 1e-6, pos, cs)
    _, n = O.add_rmsnorm(dt, q.reshape(T * H, D), np.zeros((T * H, D), np.uint16), qw, 1e-6)
    return o, n.reshape(T, H, D), cs


@pytest.mark.parametrize("rope_dim", [16, 32, 64, 128])
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_partial_rotary_nope_part_is_the_norm(dt, rope_dim):
    """The first head_dim - rope_dim elements are the per-head RMSNorm of the
    row oracle (zero residual), unrotated, at every position."""
    q, qw, pos, _ = _setup(dt, T=48)
    o, n, _ = _partial(dt, q, qw, rope_dim, pos)
    nope = D - rope_dim
    assert np.array_equal(o[..., :nope], n[..., :nope])


@pytest.mark.parametrize("rope_dim", [16, 64])
def test_partial_rotary_position_zero_is_norm_only(rope_dim):
    q, qw, pos, _ = _setup("bf16", T=24)
    o, n, _ = _partial("bf16", q, qw, rope_dim, np.zeros(24, np.int32))
    assert np.array_equal(o, n)


@pytest.mark.parametrize("rope_dim", [16, 32, 64])
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_partial_rotary_within_rounding_of_float64(dt, rope_dim):
    """The rope part: pairs (j, j + rope_dim/2) of the last rope_dim elements
    rotated by the angles of frequency j - nope (theta^(-2i/rope_dim)),
    recomputed in float64 from the rounded norm."""
    q, qw, pos, _ = _setup(dt, T=64)
    o, n, cs = _partial(dt, q, qw, rope_dim, pos)
    nope, half = D - rope_dim, rope_dim // 2
    nv = pins.bits_to_f64(n, dt)
    c = cs[pos][:, None, :half].astype(np.float64)
    s = cs[pos][:, None, half:].astype(np.float64)
    lo, hi = nv[..., nope:nope + half], nv[..., nope + half:]
    ref = np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)
    ov = pins.bits_to_f64(o[..., nope:], dt)
    mag = np.concatenate([np.abs(lo * c) + np.abs(hi * s), np.abs(hi * c) + np.abs(lo * s)], axis=-1)
    tol = 0.5 * pins.ulp(ref, dt) + 2.0 ** -22 * mag
    assert np.all(np.abs(ov - ref) <= tol)
    # and the rotation is not the identity away from position 0
    assert not np.array_equal(o[1:, :, nope:], n[1:, :, nope:])


def test_partial_rotary_of_the_whole_head_is_the_full_call():
    q, qw, pos, cs = _setup("bf16", T=40)
    T, H = q.shape[:2]
    o1 = O.qk_rmsnorm_rope("bf16", q.reshape(-1), H * D, T, H, D, qw, 1e-6, pos, cs)
    o2 = O.qk_rmsnorm_rope_partial("bf16", q.reshape(-1), H * D, T, H, D, D, qw, 1e-6, pos, cs)
    assert np.array_equal(o1, o2)


def test_partial_rotary_preserves_pair_norm():
    q, qw, pos, _ = _setup("bf16", T=128)
    o, n, _ = _partial("bf16", q, qw, 64, pos)
    nv, ov = pins.bf16_bits_to_f64(n), pins.bf16_bits_to_f64(o)
    rn = np.hypot(nv[..., 64:96], nv[..., 96:])
    ro = np.hypot(ov[..., 64:96], ov[..., 96:])
    assert np.all(np.abs(ro - rn) <= 2.0 ** -7 * rn + 1e-30)
