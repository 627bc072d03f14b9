"""GPU parity of the fused residual add + RMSNorm + FP8 / NVFP4 calls against
the CPU oracle, through the C ABI (the binding only marshals pointers)."""
import numpy as np
import pytest
import torch

import nvfp4_quant_gb300 as rq
from nvfp4_quant_gb300 import RQ_MAX_HIDDEN
import oracle as O
import synth
from nvfp4_quant_gb300 import build as rq_build
from tests import pins
from tests.gpu_util import (Guarded, assert_codes, assert_norm_within_ulp, assert_nvfp4,
                            dev16, f32dev, host8, host16)

pytestmark = pytest.mark.gpu
SMS = None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global SMS
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    rq_build.build()
    rq.lib()
    SMS = torch.cuda.get_device_properties(0).multi_processor_count


def run_fp8(dt, x, r, w, eps, scale, norm_out=True, in_place=False):
    rows, hidden = x.shape
    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    xd, rd, wd = dev16(x, dt), dev16(r, dt), dev16(w, dt)
    ro = None if in_place else Guarded((rows, hidden), tdt)
    q = Guarded((rows, hidden), torch.uint8)
    y = Guarded((rows, hidden), tdt) if norm_out else None
    rq.rq_add_rmsnorm_fp8(xd, rd, rd if in_place else ro.t, wd, eps, f32dev(scale), q.t,
                          y.t if y else None)
    torch.cuda.synchronize()
    for g in (ro, q, y):
        assert g is None or g.guards_intact(), "a kernel wrote outside its output"
    s_out = host16(rd if in_place else ro.t)
    return s_out, (host16(y.t) if y else None), host8(q.t)


def run_nvfp4(dt, x, r, w, eps, gs, norm_out=True, in_place=False):
    rows, hidden = x.shape
    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    xd, rd, wd = dev16(x, dt), dev16(r, dt), dev16(w, dt)
    ro = None if in_place else Guarded((rows, hidden), tdt)
    p = Guarded((rows, hidden // 2), torch.uint8)
    sf = Guarded((rows, hidden // 16), torch.uint8)
    y = Guarded((rows, hidden), tdt) if norm_out else None
    rq.rq_add_rmsnorm_nvfp4(xd, rd, rd if in_place else ro.t, wd, eps, f32dev(gs), p.t, sf.t,
                            y.t if y else None)
    torch.cuda.synchronize()
    for g in (ro, p, sf, y):
        assert g is None or g.guards_intact(), "a kernel wrote outside its output"
    s_out = host16(rd if in_place else ro.t)
    return s_out, (host16(y.t) if y else None), host8(p.t), host8(sf.t)


def check_fp8(dt, x, r, w, eps, scale, norm_out=True, in_place=False):
    s_ref, y_ref, q_ref = O.add_rmsnorm_fp8(dt, x, r, w, eps, scale)
    s, y, q = run_fp8(dt, x, r, w, eps, scale, norm_out, in_place)
    assert np.array_equal(s, s_ref), "residual' must be bit-exact"
    assert_codes(q, q_ref, 0x80, "FP8 codes")
    if y is not None:
        assert_norm_within_ulp(y, y_ref, dt)
        # the quantiser is exact: codes = oracle quantiser of the kernel's own y
        assert np.array_equal(q, O.quant_fp8(dt, y, scale))
    return s, y, q


def check_nvfp4(dt, x, r, w, eps, gs, norm_out=True, in_place=False):
    s_ref, y_ref, p_ref, sf_ref = O.add_rmsnorm_nvfp4(dt, x, r, w, eps, gs)
    s, y, p, sf = run_nvfp4(dt, x, r, w, eps, gs, norm_out, in_place)
    assert np.array_equal(s, s_ref), "residual' must be bit-exact"
    assert_nvfp4(p, sf, p_ref, sf_ref, y_ref, gs, dt)
    if y is not None:
        assert_norm_within_ulp(y, y_ref, dt)
        p_o, sf_o = O.quant_nvfp4(dt, y, gs)
        assert np.array_equal(sf, sf_o) and np.array_equal(p, p_o)
    return s, y, p, sf


def oracle_gs(dt, x, r, w, eps):
    _, y = O.add_rmsnorm(dt, x, r, w, eps)
    return O.nvfp4_gs_from_amax(O.amax(dt, y)), O.fp8_scale_from_amax(O.amax(dt, y))


# ------------------------------------------------------------- the five workloads
def test_tiny_fp8_16x128_bf16():
    x, r, w = synth.rows_input(0, 16, 128, "bf16")
    check_fp8("bf16", x, r, w, 1e-6, 0.05)


def test_nvfp4_tail_64x8192_fp16_with_norm_out():
    x, r, w = synth.rows_input(0, 64, 8192, "fp16")
    gs, _ = oracle_gs("fp16", x, r, w, 1e-6)
    check_nvfp4("fp16", x, r, w, 1e-6, gs, norm_out=True)


def test_prefill_fp8_65536x1024_bf16():
    x, r, w = synth.rows_input(0, 65536, 1024, "bf16", res_std=2.0)
    _, scale = oracle_gs("bf16", x, r, w, 1e-6)
    check_fp8("bf16", x, r, w, 1e-6, scale, norm_out=False, in_place=True)


def test_large_nvfp4_16384x7168_bf16_outliers_with_norm_out():
    x, r, w = synth.rows_input(0, 16384, 7168, "bf16", outlier_frac=0.01)
    gs, _ = oracle_gs("bf16", x, r, w, 1e-6)
    check_nvfp4("bf16", x, r, w, 1e-6, gs, norm_out=True, in_place=True)


# ------------------------------------------------------------- the pages' grid
@pytest.mark.parametrize("hidden", [128, 7168])
@pytest.mark.parametrize("rows", [16, 256, 8192])
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_validation_grid_nvfp4_out(hidden, rows, dt):
    x, r, w = synth.rows_input(rows + hidden, rows, hidden, dt)
    gs, _ = oracle_gs(dt, x, r, w, 1e-6)
    check_nvfp4(dt, x, r, w, 1e-6, gs, norm_out=True)


# ------------------------------------------------------------- every launch shape, ragged
# hidden sizes hit each thread-group shape, with full and partial vectors per
# thread; rows straddle the persistent grid (multiples of the SM count +- 1)
HIDDEN = [16, 48, 112, 128, 144, 496, 512, 528, 1024, 1040, 2048, 2064, 4096, 4112,
          7168, 7184, 8192, 8208, 16384, 16400, 32768]


@pytest.mark.parametrize("hidden", HIDDEN)
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_every_shape_fp8(hidden, dt):
    rows = max(1, min(3 * SMS + 1, (1 << 21) // hidden))
    x, r, w = synth.rows_input(hidden, rows, hidden, dt, res_std=2.0)
    _, scale = oracle_gs(dt, x, r, w, 1e-6)
    check_fp8(dt, x, r, w, 1e-6, scale, norm_out=True)


@pytest.mark.parametrize("hidden", HIDDEN)
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_every_shape_nvfp4(hidden, dt):
    rows = max(1, min(2 * SMS - 1, (1 << 21) // hidden))
    x, r, w = synth.rows_input(hidden + 1, rows, hidden, dt, outlier_frac=0.01)
    gs, _ = oracle_gs(dt, x, r, w, 1e-6)
    check_nvfp4(dt, x, r, w, 1e-6, gs, norm_out=(hidden % 32 == 0))


@pytest.mark.parametrize("rows", [1, 2, 3, 7, 151, 152, 153, 1217])
def test_row_counts(rows):
    x, r, w = synth.rows_input(rows, rows, 1024, "bf16")
    gs, scale = oracle_gs("bf16", x, r, w, 1e-6)
    check_fp8("bf16", x, r, w, 1e-6, scale)
    check_nvfp4("bf16", x, r, w, 1e-6, gs, in_place=True)


# ------------------------------------------------------------- edge cases
def test_zero_rows_launch_nothing():
    x = torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((0, 128), dtype=torch.uint8, device="cuda")
    w = torch.ones(128, dtype=torch.bfloat16, device="cuda")
    rq.rq_add_rmsnorm_fp8(x, x, x, w, 1e-6, f32dev(1.0), q)
    torch.cuda.synchronize()


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_zero_and_constant_rows(dt):
    H = 1024
    x = np.zeros((8, H), np.uint16)
    r = np.zeros_like(x)
    x[1] = pins.f64_to_dt(np.full(H, 0.75), dt)
    x[2] = pins.f64_to_dt(np.full(H, -3.0), dt)
    x[3, ::2] = 0x8000  # negative zeros
    _, _, w = synth.rows_input(5, 1, H, dt)
    check_fp8(dt, x, r, w, 1e-6, 0.01)
    _, y, p, sf = check_nvfp4(dt, x, r, w, 1e-6, 100.0)
    assert np.all(sf[0] == 0) and np.all(p[0] & 0x77 == 0)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_saturation_and_tiny_values(dt):
    """Outliers that saturate FP8 at 448 and rows whose blocks get subnormal
    or zero NVFP4 scales."""
    H = 2048
    x, r, w = synth.rows_input(6, 64, H, dt)
    xv = pins.bits_to_f64(x, dt)
    xv[::3, ::97] *= 300.0
    xv[1::3, 16:64] *= 1e-4
    x = pins.f64_to_dt(xv, dt)
    check_fp8(dt, x, r, w, 1e-6, 0.002)  # many |y| / scale above 448
    check_nvfp4(dt, x, r, w, 1e-6, 4000.0)


def test_power_of_two_rows_zero_eps_exact():
    """eps = 0 and rows of +-2^k: every step is exact, so the kernel matches
    the oracle bit for bit in every output."""
    H = 4096
    rng = np.random.default_rng(7)
    xv = rng.choice([-1.0, 1.0], (32, H)) * (2.0 ** rng.integers(-8, 8, 32))[:, None]
    x = pins.f64_to_bf16_carry(xv)
    r = np.zeros_like(x)
    _, _, w = synth.rows_input(7, 1, H, "bf16")
    s_ref, y_ref, q_ref = O.add_rmsnorm_fp8("bf16", x, r, w, 0.0, 0.01)
    s, y, q = run_fp8("bf16", x, r, w, 0.0, 0.01)
    assert np.array_equal(y, y_ref) and np.array_equal(q, q_ref)
    s_ref, y_ref, p_ref, sf_ref = O.add_rmsnorm_nvfp4("bf16", x, r, w, 0.0, 300.0)
    s, y, p, sf = run_nvfp4("bf16", x, r, w, 0.0, 300.0)
    assert np.array_equal(y, y_ref) and np.array_equal(p, p_ref) and np.array_equal(sf, sf_ref)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_conversions_over_every_dtype_value(dt):
    """Rows of +-1 with eps = 0 give y = w exactly, so putting every finite
    dtype value in the weight runs the kernel's E4M3 and E2M1 conversions
    (rounding, ties, saturation, signed zeros, subnormals) over all of them;
    the codes must equal the oracle's bit for bit."""
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = pins.bits_to_f64(b, dt)
    vals = b[np.isfinite(v)]
    H = 8192
    vals = np.concatenate([vals, np.zeros((-vals.size) % H, np.uint16)])
    for c in range(0, vals.size, H):
        w = vals[c:c + H]
        x = pins.f64_to_dt(np.array([[1.0] * H, [-1.0] * H]), dt)
        r = np.zeros_like(x)
        for scale in (1.0, 0.37):
            s_ref, y_ref, q_ref = O.add_rmsnorm_fp8(dt, x, r, w, 0.0, scale)
            s, y, q = run_fp8(dt, x, r, w, 0.0, scale)
            assert np.array_equal(y, y_ref)
            assert np.array_equal(q, q_ref), "E4M3 conversion differs from the oracle"
        for gs in (1.0, 0.001, 3.3e4):
            _, y_ref, p_ref, sf_ref = O.add_rmsnorm_nvfp4(dt, x, r, w, 0.0, gs)
            _, y, p, sf = run_nvfp4(dt, x, r, w, 0.0, gs)
            assert np.array_equal(sf, sf_ref), "block scale differs from the oracle"
            assert np.array_equal(p, p_ref), "E2M1 conversion differs from the oracle"


def test_out_of_place_and_in_place_agree():
    x, r, w = synth.rows_input(8, 300, 7168, "bf16")
    gs, _ = oracle_gs("bf16", x, r, w, 1e-6)
    a = run_nvfp4("bf16", x, r, w, 1e-6, gs, in_place=False)
    b = run_nvfp4("bf16", x, r, w, 1e-6, gs, in_place=True)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_norm_out_does_not_change_codes():
    x, r, w = synth.rows_input(9, 500, 1024, "fp16")
    gs, scale = oracle_gs("fp16", x, r, w, 1e-6)
    assert np.array_equal(run_fp8("fp16", x, r, w, 1e-6, scale, True)[2],
                          run_fp8("fp16", x, r, w, 1e-6, scale, False)[2])
    a = run_nvfp4("fp16", x, r, w, 1e-6, gs, True)
    b = run_nvfp4("fp16", x, r, w, 1e-6, gs, False)
    assert np.array_equal(a[2], b[2]) and np.array_equal(a[3], b[3])


def test_results_repeat_bit_for_bit():
    x, r, w = synth.rows_input(10, 2000, 2048, "bf16")
    runs = [run_nvfp4("bf16", x, r, w, 1e-6, 500.0) for _ in range(3)]
    for u in runs[1:]:
        for a, b in zip(runs[0], u):
            assert np.array_equal(a, b)


# ------------------------------------------------------------- calibration
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("hidden", [128, 1024, 7168])
def test_amax_and_scales(dt, hidden):
    x, r, w = synth.rows_input(11, 777, hidden, dt, outlier_frac=0.01)
    _, y_ref = O.add_rmsnorm(dt, x, r, w, 1e-6)
    a_ref = O.amax(dt, y_ref)
    amax = torch.full((1,), 123.0, dtype=torch.float32, device="cuda")
    rq.rq_add_rmsnorm_amax(dev16(x, dt), dev16(r, dt), dev16(w, dt), 1e-6, amax)
    a = float(amax.item())
    assert abs(a - a_ref) <= pins.ulp(np.array([a_ref]), dt)[0]
    # the scales from a given amax are one IEEE division: exact
    ad = f32dev(a_ref)
    out = f32dev(0.0)
    rq.rq_fp8_scale_from_amax(ad, out)
    assert float(out.item()) == O.fp8_scale_from_amax(a_ref)
    rq.rq_nvfp4_global_scale_from_amax(ad, out)
    assert float(out.item()) == O.nvfp4_gs_from_amax(a_ref)


def test_streams_are_honoured():
    x, r, w = synth.rows_input(12, 4096, 1024, "bf16")
    _, y_ref, q_ref = O.add_rmsnorm_fp8("bf16", x, r, w, 1e-6, 0.02)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        xd, rd, wd = dev16(x, "bf16"), dev16(r, "bf16"), dev16(w, "bf16")
        q = torch.empty((4096, 1024), dtype=torch.uint8, device="cuda")
        rq.rq_add_rmsnorm_fp8(xd, rd, rd, wd, 1e-6, f32dev(0.02), q, stream=s)
    s.synchronize()
    assert_codes(host8(q), q_ref, 0x80, "FP8 codes on a side stream")


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_fp8_codes_exact_for_every_value_at_many_scales(dt):
    """The kernels form y / scale with Markstein's correction step (or div.rn
    for divisors out of its range); the codes must equal the oracle's IEEE
    quotient for every finite dtype value, at any scale."""
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = pins.bits_to_f64(b, dt)
    vals = b[np.isfinite(v)]
    H = 8192
    vals = np.concatenate([vals, np.zeros((-vals.size) % H, np.uint16)]).reshape(-1, H)
    rng = np.random.default_rng(123)
    scales = np.exp(rng.uniform(np.log(1e-6), np.log(1e4), 48)).astype(np.float32)
    ones = pins.f64_to_dt(np.ones((1, H)), dt)
    for scale in scales:
        for w in vals:
            s_ref, y_ref, q_ref = O.add_rmsnorm_fp8(dt, ones, np.zeros_like(ones), w, 0.0, float(scale))
            _, y, q = run_fp8(dt, ones, np.zeros_like(ones), w, 0.0, float(scale), norm_out=True)
            assert np.array_equal(y, y_ref)
            assert np.array_equal(q, q_ref), "E4M3 codes differ at scale %r" % float(scale)


# ------------------------------------------------------------- long rows (staged / two-pass)
@pytest.mark.parametrize("hidden", [8208, 16384, 16400, 20480, 28672])
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_long_rows_through_shared_memory(hidden, dt):
    """Rows above 8192 elements, at least two per SM: up to 16384 elements
    the kernel that stages x and residual in shared memory, above it the
    two-pass kernel.  FP8, NVFP4, per-token FP8 and the amax calibration
    against the oracle."""
    rows = 2 * SMS + 3
    x, r, w = synth.rows_input(hidden + 7, rows, hidden, dt, res_std=2.0, outlier_frac=0.01)
    gs, scale = oracle_gs(dt, x, r, w, 1e-6)
    check_fp8(dt, x, r, w, 1e-6, scale, norm_out=True)
    check_nvfp4(dt, x, r, w, 1e-6, gs, norm_out=True, in_place=True)
    _, y_ref = O.add_rmsnorm(dt, x, r, w, 1e-6)
    xd, rd, wd = dev16(x, dt), dev16(r, dt), dev16(w, dt)
    q = torch.empty((rows, hidden), dtype=torch.uint8, device="cuda")
    sc = torch.empty(rows, dtype=torch.float32, device="cuda")
    y = torch.empty_like(xd)
    rq.rq_add_rmsnorm_fp8_per_token(xd, rd, torch.empty_like(rd), wd, 1e-6, q, sc, y)
    amax = f32dev(0.0)
    rq.rq_add_rmsnorm_amax(xd, rd, wd, 1e-6, amax)
    torch.cuda.synchronize()
    q_o, sc_o = O.quant_fp8_per_row(dt, host16(y))
    assert np.array_equal(host8(q), q_o) and np.array_equal(sc.cpu().numpy(), sc_o)
    assert_norm_within_ulp(host16(y), y_ref, dt)
    a_ref = O.amax(dt, y_ref)
    assert abs(float(amax.item()) - a_ref) <= pins.ulp(np.array([a_ref]), dt)[0]


# ------------------------------------------------------------- rows above 32768
@pytest.mark.parametrize("hidden,rows", [(32784, -2), (40976, 5), (65536, -1), (RQ_MAX_HIDDEN, 3)])
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_rows_beyond_the_register_shapes(hidden, rows, dt):
    """Rows above 32768 elements run the two-pass kernel (one CTA per row,
    residual' read back from where pass 1 stored it): FP8, NVFP4 with norm
    out, per-token FP8 and the amax calibration against the oracle.  Row
    counts -1 / -2: the SM count + 1 / twice it + 3 (past the persistent
    grid)."""
    rows = {-1: SMS + 1, -2: 2 * SMS + 3}.get(rows, rows)
    x, r, w = synth.rows_input(hidden + 9, rows, hidden, dt, res_std=2.0, outlier_frac=0.01)
    gs, scale = oracle_gs(dt, x, r, w, 1e-6)
    check_fp8(dt, x, r, w, 1e-6, scale, norm_out=True)
    check_nvfp4(dt, x, r, w, 1e-6, gs, norm_out=True, in_place=True)
    _, y_ref = O.add_rmsnorm(dt, x, r, w, 1e-6)
    xd, rd, wd = dev16(x, dt), dev16(r, dt), dev16(w, dt)
    q = torch.empty((rows, hidden), dtype=torch.uint8, device="cuda")
    sc = torch.empty(rows, dtype=torch.float32, device="cuda")
    y = torch.empty_like(xd)
    rq.rq_add_rmsnorm_fp8_per_token(xd, rd, torch.empty_like(rd), wd, 1e-6, q, sc, y)
    amax = f32dev(0.0)
    rq.rq_add_rmsnorm_amax(xd, rd, wd, 1e-6, amax)
    torch.cuda.synchronize()
    q_o, sc_o = O.quant_fp8_per_row(dt, host16(y))
    assert np.array_equal(host8(q), q_o) and np.array_equal(sc.cpu().numpy(), sc_o)
    assert_norm_within_ulp(host16(y), y_ref, dt)
    a_ref = O.amax(dt, y_ref)
    assert abs(float(amax.item()) - a_ref) <= pins.ulp(np.array([a_ref]), dt)[0]


# ------------------------------------------------------------- few rows
# At most one row per SM the rows go to wide groups (256 or 512 threads per
# row, 2 to 8 vectors per thread): every mode on each of those shapes, with
# ragged rows (hidden not a multiple of the group's reach) and row counts 1,
# 17 and the SM count.
FEW_HIDDEN = [2064, 4096, 4112, 7168, 8208, 12304, 16384, 16400]


@pytest.mark.parametrize("hidden", FEW_HIDDEN)
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_few_rows_wide_groups(hidden, dt):
    for rows in (1, 17, SMS):
        x, r, w = synth.rows_input(rows + hidden, rows, hidden, dt, outlier_frac=0.01)
        gs, scale = oracle_gs(dt, x, r, w, 1e-6)
        check_fp8(dt, x, r, w, 1e-6, scale, norm_out=True)
        _, y, p, sf = check_nvfp4(dt, x, r, w, 1e-6, gs, norm_out=True)
        # swizzled scales: the layout of the linear call's scales
        tdt = torch.bfloat16 if dt == "bf16" else torch.float16
        xd, rd, wd = dev16(x, dt), dev16(r, dt), dev16(w, dt)
        ro = torch.empty((rows, hidden), dtype=tdt, device="cuda")
        ps = torch.empty((rows, hidden // 2), dtype=torch.uint8, device="cuda")
        ss = torch.full((rq.rq_nvfp4_swizzled_scale_bytes(rows, hidden),), 0xA5, dtype=torch.uint8,
                        device="cuda")
        rq.rq_add_rmsnorm_nvfp4_swizzled(xd, rd, ro, wd, 1e-6, f32dev(gs), ps, ss)
        torch.cuda.synchronize()
        assert np.array_equal(host8(ps), p)
        assert np.array_equal(host8(ss), O.nvfp4_swizzle_scales(sf, hidden))
        # per-token FP8: codes and scales are the oracle's quantiser of y
        q = torch.empty((rows, hidden), dtype=torch.uint8, device="cuda")
        sc = torch.empty((rows,), dtype=torch.float32, device="cuda")
        rq.rq_add_rmsnorm_fp8_per_token(xd, rd, ro, wd, 1e-6, q, sc)
        torch.cuda.synchronize()
        q_o, sc_o = O.quant_fp8_per_row(dt, y)
        assert np.array_equal(host8(q), q_o) and np.array_equal(sc.cpu().numpy(), sc_o)
        # calibration: the maximum of |y|
        am = torch.empty((1,), dtype=torch.float32, device="cuda")
        rq.rq_add_rmsnorm_amax(xd, rd, wd, 1e-6, am)
        torch.cuda.synchronize()
        assert float(am.item()) == O.amax(dt, y)
