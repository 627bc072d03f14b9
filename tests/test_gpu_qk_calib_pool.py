"""GPU parity of the Q/K calibration (max |o|), dynamic-scale and mixed
KV-pool calls against the oracle, through the C ABI.

o is the dtype-rounded output of the per-head RMSNorm + NeoX RoPE.  The
kernel and the oracle sum the squares of a head in different fp32 orders, so
a norm value may differ by one dtype ulp where it sits next to a rounding
boundary: the maxima are compared within one ulp, the FP8 codes with the
usual bar (at least 99.9 % identical, never more than one step apart), and
the dtype values of the mixed pool at least 99.9 % identical and each the
rotation of a norm output within one ulp of the oracle's.
"""
import numpy as np
import pytest
import torch

import nvfp4_quant_gb300 as rq
import oracle as O
import synth
from nvfp4_quant_gb300 import build as rq_build
from tests import pins
from tests.gpu_util import assert_codes, dev16, f32dev, host8

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    rq_build.build()
    rq.lib()


def _dev_i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def oracle_o(dt, x, w, pos, cs, rope_dim=D):
    T, H = x.shape[:2]
    if rope_dim == D:
        return O.qk_rmsnorm_rope(dt, x.reshape(-1), H * D, T, H, D, w, 1e-6, pos, cs)
    return O.qk_rmsnorm_rope_partial(dt, x.reshape(-1), H * D, T, H, D, rope_dim, w, 1e-6, pos, cs)


def assert_amax(got, o_ref, dt):
    ref = O.amax(dt, o_ref)
    ulp = float(pins.ulp(np.array([ref]), dt)[0])
    assert abs(got - ref) <= ulp, "amax %r against the oracle's %r" % (got, ref)


@pytest.mark.parametrize("T,Hq,Hk,dt", [(4096, 16, 8, "bf16"), (1, 3, 1, "bf16"), (333, 5, 3, "fp16"),
                                        (1000, 16, 0, "bf16"), (77, 0, 4, "fp16")])
def test_qk_amax(T, Hq, Hk, dt):
    q, k, qw, kw, pos, cs = synth.qk_input(T + Hq, T, max(Hq, 1), max(Hk, 1), D, dt)
    q, k = q[:, :Hq], k[:, :Hk]
    qa = torch.full((1,), 123.0, device="cuda")
    ka = torch.full((1,), 456.0, device="cuda")
    rq.rq_qk_rmsnorm_rope_amax(dev16(q, dt) if Hq else None, dev16(k, dt) if Hk else None,
                               dev16(qw, dt), dev16(kw, dt), 1e-6, _dev_i32(pos),
                               torch.from_numpy(cs).cuda(), qa, ka)
    torch.cuda.synchronize()
    if Hq:
        assert_amax(qa.item(), oracle_o(dt, q, qw, pos, cs), dt)
    else:
        assert qa.item() == 123.0  # a side without heads is left alone
    if Hk:
        assert_amax(ka.item(), oracle_o(dt, k, kw, pos, cs), dt)
    else:
        assert ka.item() == 456.0


def test_qk_amax_shared_address_and_empty():
    T, Hq, Hk = 200, 4, 2
    q, k, qw, kw, pos, cs = synth.qk_input(3, T, Hq, Hk, D, "bf16")
    a = torch.full((1,), -1.0, device="cuda")
    rq.rq_qk_rmsnorm_rope_amax(dev16(q, "bf16"), dev16(k, "bf16"), dev16(qw, "bf16"),
                               dev16(kw, "bf16"), 1e-6, _dev_i32(pos), torch.from_numpy(cs).cuda(),
                               a, a)
    torch.cuda.synchronize()
    both = np.concatenate([oracle_o("bf16", q, qw, pos, cs).ravel(),
                           oracle_o("bf16", k, kw, pos, cs).ravel()])
    assert_amax(a.item(), both, "bf16")
    # an empty call clears the maximum
    e = torch.zeros((0, Hq, D), dtype=torch.bfloat16, device="cuda")
    rq.rq_qk_rmsnorm_rope_amax(e, None, dev16(qw, "bf16"), None, 1e-6, _dev_i32(pos[:0]),
                               torch.from_numpy(cs).cuda(), a, None)
    torch.cuda.synchronize()
    assert a.item() == 0.0


@pytest.mark.parametrize("T,Hq,Hk,dt", [(4096, 16, 8, "bf16"), (500, 6, 2, "fp16")])
def test_qk_dynamic_scales(T, Hq, Hk, dt):
    """Scales amax(o) / 448 of the call's own maxima; codes against the
    oracle's quantiser at the oracle's scales; no code beyond 448 except the
    maxima themselves."""
    q, k, qw, kw, pos, cs = synth.qk_input(11, T, Hq, Hk, D, dt)
    qs, ks = torch.zeros(1, device="cuda"), torch.zeros(1, device="cuda")
    qo = torch.empty((T, Hq, D), dtype=torch.uint8, device="cuda")
    ko = torch.empty((T, Hk, D), dtype=torch.uint8, device="cuda")
    args = (dev16(q, dt), dev16(k, dt), dev16(qw, dt), dev16(kw, dt), 1e-6, _dev_i32(pos),
            torch.from_numpy(cs).cuda())
    rq.rq_qk_rmsnorm_rope_fp8_dynamic(*args, qs, ks, qo, ko)
    qa, ka = torch.zeros(1, device="cuda"), torch.zeros(1, device="cuda")
    rq.rq_qk_rmsnorm_rope_amax(*args, qa, ka)
    torch.cuda.synchronize()
    # the scales are the plain formula on the call's own maxima, bit for bit
    assert qs.item() == O.fp8_dynamic_scale(qa.item())
    assert ks.item() == O.fp8_dynamic_scale(ka.item())
    for x, w, s_dev, codes, what in ((q, qw, qs, qo, "Q"), (k, kw, ks, ko, "K")):
        o = oracle_o(dt, x, w, pos, cs)
        s_ref = O.fp8_dynamic_scale(O.amax(dt, o))
        assert abs(s_dev.item() - s_ref) <= 2.0 ** -22 * s_ref
        ref = O.quant_fp8(dt, o, s_ref)
        got = host8(codes)
        assert_codes(got, ref, 0x80, what + " codes")
        # 0x7E / 0xFE is 448: only the elements at the maximum reach it
        sat = np.count_nonzero((got & 0x7F) == 0x7E)
        assert 1 <= sat <= 4, "%s: %d codes at 448" % (what, sat)


def test_qk_dynamic_zero_input():
    T, H = 16, 2
    _, _, qw, kw, pos, cs = synth.qk_input(1, T, H, H, D, "bf16")
    z = torch.zeros((T, H, D), dtype=torch.bfloat16, device="cuda")
    qs, ks = torch.zeros(1, device="cuda"), torch.zeros(1, device="cuda")
    qo = torch.full((T, H, D), 0x55, dtype=torch.uint8, device="cuda")
    ko = torch.full((T, H, D), 0x55, dtype=torch.uint8, device="cuda")
    rq.rq_qk_rmsnorm_rope_fp8_dynamic(z, z, dev16(qw, "bf16"), dev16(kw, "bf16"), 1e-6,
                                      _dev_i32(pos), torch.from_numpy(cs).cuda(), qs, ks, qo, ko)
    torch.cuda.synchronize()
    assert qs.item() == 1.0 and ks.item() == 1.0
    # every code a zero; its sign is the rotation's (+0 * c - (+0) * s can be -0)
    zero_bits = np.zeros((T, H, D), np.uint16)
    for codes in (qo, ko):
        got = host8(codes)
        assert not (got & 0x7F).any()
        assert np.array_equal(got, O.quant_fp8("bf16", oracle_o("bf16", zero_bits, qw, pos, cs), 1.0))


def run_mixed(dt, q, k, qw, kw, pos, cs, qscale, kscale, slots, n_slots, rope_dim):
    T, Hq, Hk = q.shape[0], q.shape[1], k.shape[1]
    pool = torch.full((n_slots, Hk, D + rope_dim), 0x5A, dtype=torch.uint8, device="cuda")
    qo = torch.empty((T, Hq, D), dtype=torch.uint8, device="cuda")
    rq.rq_qk_rmsnorm_rope_fp8_kv_store_mixed(dev16(q, dt), dev16(k, dt), dev16(qw, dt),
                                             dev16(kw, dt), 1e-6, _dev_i32(pos),
                                             torch.from_numpy(cs).cuda(), f32dev(qscale),
                                             f32dev(kscale), qo, pool,
                                             torch.from_numpy(slots).cuda(), rope_dim)
    torch.cuda.synchronize()
    return host8(qo), host8(pool)


def _rot_candidates(n_lo, n_hi, c, s, dt):
    """dt(RN32(RN32(n_lo c) - RN32(n_hi s))) and dt(RN32(RN32(n_hi c) +
    RN32(n_lo s))) as float64 values, the steps in fp32 (numpy float32
    arithmetic is IEEE round to nearest)."""
    f = np.float32
    lo = (f(n_lo) * f(c)) - (f(n_hi) * f(s))
    hi = (f(n_hi) * f(c)) + (f(n_lo) * f(s))
    rd = lambda v: pins.bits_to_f64(synth.to_bits(np.asarray(v, np.float64), dt), dt)
    return rd(lo), rd(hi)


def _neighbours(bits):
    """The dtype values (float64) of a bit pattern and of the patterns one
    step below and above it on the number line."""
    b = int(bits)
    o = -(b & 0x7FFF) if b & 0x8000 else b & 0x7FFF  # ordinal, +0 and -0 both 0
    out = []
    for d in (-1, 0, 1):
        m = o + d
        out.append(((-m) | 0x8000) if m < 0 else m)
    return out


def assert_rotation(rope, rope_ref, x, w, pos, cs, dt):
    """The rope values: at least 99.9 % identical to the oracle's, and each
    one the rotation (the oracle's fp32 steps) of a norm output within one
    ulp of the oracle's.  (The sum-of-squares order may move a norm value by
    one ulp; where the rotation cancels, that is more than one ulp of the
    rotated value.)"""
    same = rope == rope_ref
    assert np.mean(same) >= 0.999, "rope values: only %.5f identical" % np.mean(same)
    if same.all():
        return
    R = rope.shape[-1]
    half = R // 2
    # the oracle's norm output of the heads
    n_all = O.add_rmsnorm(dt, x.reshape(-1, D), np.zeros((x.size // D, D), np.uint16), w, 1e-6)[1]
    n_all = n_all.reshape(x.shape)[..., D - R:]
    got = pins.bits_to_f64(rope, dt)
    for t, h, j in zip(*np.nonzero(~same)):
        i = j % half
        c, s = cs[pos[t], i], cs[pos[t], half + i]
        los = pins.bits_to_f64(np.array(_neighbours(n_all[t, h, i]), np.uint16), dt)
        his = pins.bits_to_f64(np.array(_neighbours(n_all[t, h, half + i]), np.uint16), dt)
        cands = []
        for l2 in los:
            for h2 in his:
                o_lo, o_hi = _rot_candidates(l2, h2, c, s, dt)
                cands.append(float(np.ravel(o_lo if j < half else o_hi)[0]))
        assert got[t, h, j] in cands, (
            "rope value (%d, %d, %d) = %r is no rotation of a norm within one ulp: oracle %r, "
            "candidates %r" % (t, h, j, got[t, h, j], pins.bits_to_f64(rope_ref[t, h, j], dt), cands))


def check_mixed(dt, T, Hq, Hk, rope_dim, seed):
    q, k, qw, kw, pos, _ = synth.qk_input(seed, T, Hq, Hk, D, dt)
    cs = synth.rope_cos_sin(T, rope_dim, 1.0e6)
    n_slots = 2 * T + 5
    rng = np.random.default_rng(seed)
    slots = rng.permutation(n_slots)[:T].astype(np.int64)
    slots[::13] = -1  # padding tokens
    if T > 5:
        slots[5] = n_slots + 1  # beyond the pool: nothing stored
    oq = oracle_o(dt, q, qw, pos, cs, rope_dim)
    ok_ = oracle_o(dt, k, kw, pos, cs, rope_dim)
    qs = O.fp8_scale_from_amax(O.amax(dt, oq))
    ks = O.fp8_scale_from_amax(O.amax(dt, ok_[..., :D - rope_dim])) if rope_dim < D else 1.0
    qo, pool = run_mixed(dt, q, k, qw, kw, pos, cs, qs, ks, slots, n_slots, rope_dim)
    assert_codes(qo, O.quant_fp8(dt, oq, qs), 0x80, "Q codes")
    nope = D - rope_dim
    written = (slots >= 0) & (slots < n_slots)
    untouched = np.ones(n_slots, bool)
    untouched[slots[written]] = False
    assert np.all(pool[untouched] == 0x5A), "a pool row outside the slots was written"
    rows = pool[slots[written]]                     # [n, Hk, D + rope_dim]
    ref = ok_[written]                              # [n, Hk, D] dtype bits
    if nope:
        assert_codes(rows[..., :nope], O.quant_fp8(dt, np.ascontiguousarray(ref[..., :nope]), ks),
                     0x80, "K nope codes")
    rope = np.ascontiguousarray(rows[..., nope:]).view(np.uint16)
    assert_rotation(rope, ref[..., nope:], k[written], kw, pos[written], cs, dt)


def test_mixed_pool_4096_tokens_16q_8k_rope64_bf16():
    check_mixed("bf16", 4096, 16, 8, 64, seed=0)


@pytest.mark.parametrize("rope_dim", [16, 32, 64, 128])
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_mixed_pool_rope_dims(dt, rope_dim):
    check_mixed(dt, 300, 5, 3, rope_dim, seed=rope_dim)


def test_mixed_pool_rope128_is_the_uniform_rotation():
    """With the whole head rotated, Q's codes are those of the uniform call,
    bit for bit (same arithmetic), and K's pool rows hold the dtype values
    that the uniform call quantises."""
    T, Hq, Hk = 257, 8, 4
    q, k, qw, kw, pos, cs = synth.qk_input(9, T, Hq, Hk, D, "bf16")
    slots = np.arange(T, dtype=np.int64)
    qo, pool = run_mixed("bf16", q, k, qw, kw, pos, cs, 0.02, 0.03, slots, T, D)
    qo2 = torch.empty((T, Hq, D), dtype=torch.uint8, device="cuda")
    ko2 = torch.empty((T, Hk, D), dtype=torch.uint8, device="cuda")
    rq.rq_qk_rmsnorm_rope_fp8(dev16(q, "bf16"), dev16(k, "bf16"), dev16(qw, "bf16"),
                              dev16(kw, "bf16"), 1e-6, _dev_i32(pos), torch.from_numpy(cs).cuda(),
                              f32dev(0.02), f32dev(0.03), qo2, ko2)
    torch.cuda.synchronize()
    assert np.array_equal(qo, host8(qo2))
    vals = np.ascontiguousarray(pool).view(np.uint16)  # [T, Hk, D]
    assert np.array_equal(O.quant_fp8("bf16", vals, 0.03), host8(ko2))
