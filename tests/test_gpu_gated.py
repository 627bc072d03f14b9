"""GPU parity of rq_gated_rmsnorm_nvfp4 against the oracle, through the C ABI.

The gate is g = dt(x * dt(silu(z))).  The kernel forms dt(silu(z)) exactly:
a fast fp32 estimate, and a double-precision evaluation wherever that
estimate lies within its error window of a dtype rounding boundary.  Every
one of the 65,536 gates of each dtype is checked against the oracle's
(test_gate_exact_over_every_dtype_value), so the gated call meets the same
bar as the residual path: the norm output within 1 ulp (only the fp32 order
of the sum of squares differs), block scales and E2M1 codes at least 99.9 %
identical and never more than one step apart, the codes exactly the oracle's
quantiser applied to the kernel's own norm output.  Two exact checks tie the
gated path to the plain one: with z = 32 and eps = 0 it equals the residual
add path on x with a residual of -0, bit for bit, and a zero gate gives zero
rows.
"""
import numpy as np
import pytest
import torch

import nvfp4_quant_gb300 as rq
import oracle as O
import synth
from nvfp4_quant_gb300 import build as rq_build
from tests import pins
from tests.gpu_util import (Guarded, assert_norm_within_ulp, assert_nvfp4, dev16, f32dev, host8,
                            host16)

pytestmark = pytest.mark.gpu
SMS = None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global SMS
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    rq_build.build()
    rq.lib()
    SMS = torch.cuda.get_device_properties(0).multi_processor_count


def run_gated(dt, x, z, w, eps, gs, norm_out=True):
    rows, hidden = x.shape
    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    xd, zd, wd = dev16(x, dt), dev16(z, dt), dev16(w, dt)
    p = Guarded((rows, hidden // 2), torch.uint8)
    sf = Guarded((rows, hidden // 16), torch.uint8)
    y = Guarded((rows, hidden), tdt) if norm_out else None
    rq.rq_gated_rmsnorm_nvfp4(xd, zd, wd, eps, f32dev(gs), p.t, sf.t, y.t if y else None)
    torch.cuda.synchronize()
    for g in (p, sf, y):
        assert g is None or g.guards_intact(), "a kernel wrote outside its output"
    assert np.array_equal(host16(xd), x) and np.array_equal(host16(zd), z), "inputs changed"
    return (host16(y.t) if y else None), host8(p.t), host8(sf.t)


def gated_gs(dt, x, z, w, eps):
    _, y = O.gated_rmsnorm(dt, x, z, w, eps)
    return O.nvfp4_gs_from_amax(O.amax(dt, y))


def check_gated(dt, x, z, w, eps, gs):
    _, y_ref, p_ref, sf_ref = O.gated_rmsnorm_nvfp4(dt, x, z, w, eps, gs)
    y, p, sf = run_gated(dt, x, z, w, eps, gs)
    assert_norm_within_ulp(y, y_ref, dt)
    assert_nvfp4(p, sf, p_ref, sf_ref, y_ref, gs, dt)
    p_o, sf_o = O.quant_nvfp4(dt, y, gs)
    assert np.array_equal(p, p_o) and np.array_equal(sf, sf_o), "quantiser not exact"
    return y, p, sf


def test_gated_16384x7168_bf16():
    x, z, w = synth.rows_input(0, 16384, 7168, "bf16", outlier_frac=0.01)
    check_gated("bf16", x, z, w, 1e-6, gated_gs("bf16", x, z, w, 1e-6))


HIDDEN = [16, 48, 128, 144, 512, 1040, 2064, 4096, 4112, 6016, 7168, 8208, 16384, 32768, 40976]


@pytest.mark.parametrize("hidden", HIDDEN)
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_gated_every_shape(hidden, dt):
    # rows past the persistent grid, and the long-row shared-memory kernel
    # (at least two rows per SM) for 8208 and 16384
    for rows in (max(1, min(3 * SMS + 1, (1 << 21) // hidden)), 7):
        if hidden in (8208, 16384) and rows > 7:
            rows = 2 * SMS + 3
        x, z, w = synth.rows_input(hidden + rows, rows, hidden, dt, res_std=2.0)
        check_gated(dt, x, z, w, 1e-6, gated_gs(dt, x, z, w, 1e-6))


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("hidden", [1040, 7168, 16384])
def test_gate_of_32_equals_the_plain_path(dt, hidden):
    rows = 2 * SMS + 3 if hidden == 16384 else 300
    x, _, w = synth.rows_input(9, rows, hidden, dt)
    z = np.full((rows, hidden), synth.to_bits(np.array([32.0]), dt)[0], np.uint16)
    gs = 80.0
    y, p, sf = run_gated(dt, x, z, w, 0.0, gs)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    xd, wd = dev16(x, dt), dev16(w, dt)
    # a residual of -0: x + (-0) = x for every x, signed zeros included
    zero = torch.full((rows, hidden), -0.0, dtype=tdt, device="cuda")
    ro, y2 = torch.empty_like(zero), torch.empty_like(zero)
    p2 = torch.empty((rows, hidden // 2), dtype=torch.uint8, device="cuda")
    sf2 = torch.empty((rows, hidden // 16), dtype=torch.uint8, device="cuda")
    rq.rq_add_rmsnorm_nvfp4(xd, zero, ro, wd, 0.0, f32dev(gs), p2, sf2, y2)
    torch.cuda.synchronize()
    if hidden != 7168:
        # the same thread shape: the same order of the sum of squares
        assert np.array_equal(y, host16(y2)) and np.array_equal(p, host8(p2))
        assert np.array_equal(sf, host8(sf2))
    else:
        # the gated call runs these rows with more, shorter threads, so its
        # sum of squares is added in another order: 1 ulp, and each call's
        # codes exact for its own norm output
        assert_norm_within_ulp(y, host16(y2), dt)
        for yy, pp, ss in ((y, p, sf), (host16(y2), host8(p2), host8(sf2))):
            p_o, sf_o = O.quant_nvfp4(dt, yy, gs)
            assert np.array_equal(pp, p_o) and np.array_equal(ss, sf_o)


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_zero_gate_and_empty(dt):
    rows, hidden = 33, 2048
    x, _, w = synth.rows_input(10, rows, hidden, dt)
    z = np.zeros((rows, hidden), np.uint16)
    y, p, sf = run_gated(dt, x, z, w, 1e-6, 50.0)
    assert np.all(pins.bits_to_f64(y, dt) == 0.0)
    assert np.all(sf == 0) and np.all((p & 0x77) == 0)
    e = torch.zeros((0, hidden), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros((0, hidden // 2), dtype=torch.uint8, device="cuda")
    s = torch.zeros((0, hidden // 16), dtype=torch.uint8, device="cuda")
    rq.rq_gated_rmsnorm_nvfp4(e, e, torch.ones(hidden, dtype=torch.bfloat16, device="cuda"),
                              1e-6, f32dev(1.0), q, s)


def test_gate_saturates_and_handles_extreme_gates():
    # very negative gates give -0 (e^-z overflows), very positive ones pass x
    rows, hidden = 20, 256
    x, _, w = synth.rows_input(11, rows, hidden, "bf16")
    zv = np.where(np.arange(hidden) % 2 == 0, -200.0, 200.0) * np.ones((rows, 1))
    z = synth.to_bits(zv, "bf16")
    check_gated("bf16", x, z, w, 1e-6, gated_gs("bf16", x, z, w, 1e-6))


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_gates_at_and_beyond_the_table_edges(dt):
    # the 448 x 2 shape (more rows than SMs, 7168 elements), whose gates come
    # from the shared-memory tables: gates on both sides of each table's
    # edges (bf16 2^-23 and 512, fp16 32) and far beyond, mixed with N(0, 1)
    # gates in the same vectors
    rows, hidden = SMS + 48, 7168
    x, z, w = synth.rows_input(12, rows, hidden, dt)
    # (large enough to cross the edges, small enough that x * gate and the
    # sum of squares stay finite)
    edges = {"bf16": [2.0 ** -23, 2.0 ** -24, 2.0 ** -30, 508.0, 512.0, 1000.0, 3.0e4],
             "fp16": [31.96875, 32.0, 33.0, 40.0, 1000.0, 2.0 ** -24, 6.0e-5]}[dt]
    vals = np.array(edges + [-e for e in edges])
    zf = pins.bits_to_f64(z, dt)
    pick = (np.arange(rows * hidden).reshape(rows, hidden) * 7919) % 5 == 0
    zf = np.where(pick, vals[(np.arange(rows * hidden).reshape(rows, hidden) // 5) % vals.size], zf)
    z = pins.f64_to_dt(zf, dt)
    check_gated(dt, x, z, w, 1e-6, gated_gs(dt, x, z, w, 1e-6))


def test_gate_exact_over_every_dtype_value(tmp_path):
    """The kernel's gate dt(silu(z)) (tests/cuda/silu_check.cu runs the
    library's device code: the fast path with its exact path for both dtypes,
    and the shared-memory tables with their closed forms that the gated
    kernels use) for every finite bf16 and fp16 value z, bit for bit against the
    oracle's; and the fast path's error, over every finite fp32 input it
    serves, within the window of the near-tie test."""
    import os
    import subprocess
    here = os.path.dirname(os.path.abspath(__file__))
    csrc = os.path.join(os.path.dirname(here), "nvfp4_quant_gb300", "csrc")
    exe, out = str(tmp_path / "silu_check"), str(tmp_path / "gates.bin")
    subprocess.run(["nvcc", "-std=c++17", "-O3", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-I" + csrc, os.path.join(here, "cuda", "silu_check.cu"), "-o", exe], check=True)
    res = subprocess.run([exe, out], check=True, capture_output=True, text=True, timeout=600).stdout
    print(res)
    f = [l.split() for l in res.splitlines() if l.startswith("silu")][0]
    v = {f[i]: int(f[i + 1]) for i in range(1, len(f) - 1, 2)}
    assert v["max_bits"] <= v["window"], res
    gates = np.fromfile(out, np.uint16).reshape(4, 65536)
    z = np.arange(65536, dtype=np.uint16)
    for i, dt in enumerate(["bf16", "fp16", "bf16", "fp16"]):  # then the two table paths
        finite = np.isfinite(pins.bits_to_f64(z, dt))
        ref = O.silu_dt(dt, z)
        bad = np.flatnonzero(finite & (gates[i] != ref))
        assert bad.size == 0, "%s gates differ from the oracle's at z bits %s" % (
            dt, [hex(b) for b in bad[:8]])
    # among |z| <= 8, the exact path is the exception (fp16: mostly the
    # values whose SiLU is an fp16 subnormal, |z| < 2^-13)
    assert v["slow_bf16"] < 65536 // 100 and v["slow_fp16"] < 65536 // 8, res


@pytest.mark.parametrize("rows,hidden,dt", [(130, 96, "bf16"), (300, 1056, "fp16"), (16384, 7168, "bf16"),
                                            (1300, 7168, "fp16"), (-1, 16384, "bf16"), (5, 8208, "fp16")])
def test_gated_swizzled_scales(rows, hidden, dt):
    """The swizzled gated call: codes equal to the linear call's, scales byte
    for byte the oracle's layout of the linear call's scales, padding zero
    (the buffer is poisoned beforehand)."""
    rows = 2 * SMS + 3 if rows == -1 else rows
    x, z, w = synth.rows_input(rows + 3, rows, hidden, dt)
    gs = gated_gs(dt, x, z, w, 1e-6)
    _, p, sf = run_gated(dt, x, z, w, 1e-6, gs, norm_out=False)
    xd, zd, wd = dev16(x, dt), dev16(z, dt), dev16(w, dt)
    p2 = Guarded((rows, hidden // 2), torch.uint8)
    sz = Guarded((rq.rq_nvfp4_swizzled_scale_bytes(rows, hidden),), torch.uint8)
    rq.rq_gated_rmsnorm_nvfp4_swizzled(xd, zd, wd, 1e-6, f32dev(gs), p2.t, sz.t)
    torch.cuda.synchronize()
    assert p2.guards_intact() and sz.guards_intact(), "a kernel wrote outside its output"
    assert np.array_equal(host8(p2.t), p)
    assert np.array_equal(host8(sz.t), O.nvfp4_swizzle_scales(sf.reshape(rows, hidden // 16), hidden))
