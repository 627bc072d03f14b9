"""The GEMM-facing NVFP4 block-scale layout on the GPU.

1. Pin of the oracle's layout.  The pages do not print it; the consumer fixes
   it.  The oracle's packed E2M1 codes and its swizzled E4M3 scales are fed
   to cuBLASLt's block-scaled NVFP4 GEMM (through torch._scaled_mm), and the
   product must equal the fp64 product of the dequantised operands.  Layouts
   with a plausible mistake planted in them (on the CPU) must fail the same
   comparison, which shows that it sees the byte order.
2. Parity of the swizzled kernel calls: the scales of
   rq_add_rmsnorm_nvfp4_swizzled equal the oracle's swizzle of the linear
   call's scales byte for byte (padding included, in a buffer poisoned
   before the call), the other outputs equal the linear call's, and the
   kernel's swizzled output feeds the same GEMM.
"""
import numpy as np
import pytest
import torch

import nvfp4_quant_gb300 as rq
import oracle as O
import synth
from nvfp4_quant_gb300 import build as rq_build
from tests.gpu_util import Guarded, assert_codes, dev16, f32dev, host8, host16

pytestmark = pytest.mark.gpu
SMS = None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global SMS
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    rq_build.build()
    rq.lib()
    SMS = torch.cuda.get_device_properties(0).multi_processor_count


# ------------------------------------------------------------------ helpers
def spread_rows(seed, tid, rows, hidden, dt="bf16"):
    """N(0,1) rows whose 16-element blocks are scaled by 2^u, u uniform in
    -6..6, so that neighbouring block scales differ and a misplaced scale
    changes the product visibly."""
    v = synth.normal(seed, tid, rows * hidden).reshape(rows, hidden // 16, 16)
    u = np.floor(13.0 * synth.uniform(seed, tid + 1, rows * (hidden // 16))) - 6.0
    v = v * np.exp2(np.minimum(u, 6.0)).reshape(rows, hidden // 16, 1)
    return synth.to_bits(v.reshape(rows, hidden), dt)


def raw_values(packed, sf):
    """e2m1(code) * sf, float64 [rows, hidden] (the GEMM's view: no global scale)."""
    return O.nvfp4_dequant(packed, sf, 1.0)


def gemm_nvfp4(pa, sa, pb, sb):
    """cuBLASLt block-scaled NVFP4 GEMM: A [M, K] x B [N, K]^T, scales in the
    swizzled layout, bf16 out (as float64 on the host)."""
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("this torch has no packed FP4 dtype")
    a = torch.from_numpy(np.ascontiguousarray(pa)).cuda().view(torch.float4_e2m1fn_x2)
    b = torch.from_numpy(np.ascontiguousarray(pb)).cuda().view(torch.float4_e2m1fn_x2)
    sa_t = torch.from_numpy(np.ascontiguousarray(sa)).cuda().view(torch.float8_e4m3fn)
    sb_t = torch.from_numpy(np.ascontiguousarray(sb)).cuda().view(torch.float8_e4m3fn)
    try:
        c = torch._scaled_mm(a, b.t(), sa_t, sb_t, out_dtype=torch.bfloat16)
    except (RuntimeError, NotImplementedError) as e:
        pytest.skip("block-scaled NVFP4 GEMM unavailable here: %s" % str(e).splitlines()[0])
    torch.cuda.synchronize()
    return c.float().cpu().numpy().astype(np.float64)


def gemm_matches(c, ra, rb):
    """c against the fp64 product: bf16 output rounding plus fp32 accumulation."""
    ref = ra @ rb.T
    mag = np.abs(ra) @ np.abs(rb).T
    tol = 2.0 ** -8 * np.abs(ref) + 2.0 ** -14 * mag
    return bool(np.all(np.abs(c - ref) <= tol)), float(np.max(np.abs(c - ref) / (mag + 1e-30)))


def planted_layout(sf, kind):
    """The scales in a layout with one plausible mistake (CPU): 'linear' keeps
    the padded row-major matrix, 'tile_row_major' puts (r, c) at 4 r + c
    inside a tile, 'tiles_by_column' orders the tiles column of tiles first."""
    rows, nb = sf.shape
    rp, cp = -(-rows // 128) * 128, -(-nb // 4) * 4
    m = np.zeros((rp, cp), np.uint8)
    m[:rows, :nb] = sf
    if kind == "linear":
        return m.ravel()
    out = np.zeros(rp * cp, np.uint8)
    r = np.arange(rp)[:, None]
    c = np.arange(cp)[None, :]
    if kind == "tile_row_major":
        off = ((r // 128) * (cp // 4) + c // 4) * 512 + 4 * (r % 128) + c % 4
    else:
        off = ((c // 4) * (rp // 128) + r // 128) * 512 + 16 * (r % 32) + 4 * ((r % 128) // 32) + c % 4
    out[off.ravel()] = m.ravel()
    return out


def oracle_operand(seed, tid, rows, hidden):
    y = spread_rows(seed, tid, rows, hidden)
    packed, sf = O.quant_nvfp4("bf16", y, 1.0)
    return packed, sf


GEMM_SHAPES = [(130, 144, 96), (256, 128, 1024), (200, 160, 1056), (128, 256, 7168)]


@pytest.mark.parametrize("m,n,k", GEMM_SHAPES)
def test_oracle_layout_is_what_the_block_scaled_gemm_reads(m, n, k):
    pa, sfa = oracle_operand(11, 40, m, k)
    pb, sfb = oracle_operand(12, 50, n, k)
    ra, rb = raw_values(pa, sfa), raw_values(pb, sfb)
    c = gemm_nvfp4(pa, O.nvfp4_swizzle_scales(sfa, k), pb, O.nvfp4_swizzle_scales(sfb, k))
    ok, worst = gemm_matches(c, ra, rb)
    assert ok, "GEMM with the oracle's layout is off by %.3g of sum |a b|" % worst


@pytest.mark.parametrize("kind", ["linear", "tile_row_major", "tiles_by_column"])
def test_a_planted_layout_mistake_is_seen(kind):
    m, n, k = 256, 128, 1024
    pa, sfa = oracle_operand(11, 40, m, k)
    pb, sfb = oracle_operand(12, 50, n, k)
    ra, rb = raw_values(pa, sfa), raw_values(pb, sfb)
    c = gemm_nvfp4(pa, planted_layout(sfa, kind), pb, O.nvfp4_swizzle_scales(sfb, k))
    ok, _ = gemm_matches(c, ra, rb)
    assert not ok, "the GEMM comparison did not notice the %s layout" % kind


# ------------------------------------------------------------ kernel parity
def run_linear_and_swizzled(dt, x, r, w, eps, gs, dynamic=False):
    """Both layouts on the same inputs, each output in a poisoned, guarded
    buffer; returns host copies (s, y, packed, sf) for each call."""
    rows, hidden = x.shape
    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    xd, rd, wd = dev16(x, dt), dev16(r, dt), dev16(w, dt)
    outs = []
    for swz in (False, True):
        ro = Guarded((rows, hidden), tdt)
        y = Guarded((rows, hidden), tdt)
        p = Guarded((rows, hidden // 2), torch.uint8)
        nsf = rq.rq_nvfp4_swizzled_scale_bytes(rows, hidden) if swz else rows * (hidden // 16)
        sf = Guarded((nsf,), torch.uint8)
        g = torch.zeros(1, dtype=torch.float32, device="cuda") if dynamic else f32dev(gs)
        fn = {(False, False): rq.rq_add_rmsnorm_nvfp4,
              (True, False): rq.rq_add_rmsnorm_nvfp4_swizzled,
              (False, True): rq.rq_add_rmsnorm_nvfp4_dynamic,
              (True, True): rq.rq_add_rmsnorm_nvfp4_dynamic_swizzled}[(swz, dynamic)]
        fn(xd, rd, ro.t, wd, eps, g, p.t, sf.t, y.t)
        torch.cuda.synchronize()
        for b in (ro, y, p, sf):
            assert b.guards_intact(), "a kernel wrote outside its output"
        outs.append((host16(ro.t), host16(y.t), host8(p.t), host8(sf.t), float(g.item())))
    return outs


def oracle_gs(dt, x, r, w, eps):
    _, y = O.add_rmsnorm(dt, x, r, w, eps)
    return O.nvfp4_gs_from_amax(O.amax(dt, y))


STAGED = -1  # 2 * SMs + 3 rows: enough for the shared-memory kernel
CASES = [(1, 16, "bf16"), (127, 48, "fp16"), (129, 80, "bf16"), (130, 96, "bf16"),
         (300, 1056, "fp16"), (257, 7168, "bf16"), (STAGED, 8208, "bf16"),
         (STAGED, 16384, "fp16"), (3, 32768, "bf16"),
         # several rows per CTA, and a ragged last tile of 128 rows
         (2000, 7168, "bf16"), (3700, 4096, "fp16"),
         # rows above 32768 elements (the two-pass kernel)
         (5, 40976, "bf16"), (130, 65536, "fp16")]


@pytest.mark.parametrize("rows,hidden,dt", CASES)
def test_swizzled_call_matches_linear_call_and_oracle(rows, hidden, dt):
    rows = 2 * SMS + 3 if rows == STAGED else rows
    x, r, w = synth.rows_input(5, rows, hidden, dt)
    gs = oracle_gs(dt, x, r, w, 1e-6)
    (s1, y1, p1, sf1, _), (s2, y2, p2, sf2, _) = run_linear_and_swizzled(dt, x, r, w, 1e-6, gs)
    assert np.array_equal(s1, s2) and np.array_equal(y1, y2) and np.array_equal(p1, p2)
    sf1 = sf1.reshape(rows, hidden // 16)
    # every byte, padding included, is the layout of the linear call's scales
    assert np.array_equal(sf2, O.nvfp4_swizzle_scales(sf1, hidden))
    # and against the oracle's own scales, in the swizzled order
    _, _, _, sf_ref = O.add_rmsnorm_nvfp4(dt, x, r, w, 1e-6, gs)
    assert_codes(sf2, O.nvfp4_swizzle_scales(sf_ref, hidden), 0x80, "swizzled block scales")


@pytest.mark.parametrize("rows,hidden", [(300, 1056), (257, 7168)])
def test_dynamic_swizzled_call(rows, hidden):
    x, r, w = synth.rows_input(6, rows, hidden, "bf16")
    (s1, y1, p1, sf1, g1), (s2, y2, p2, sf2, g2) = run_linear_and_swizzled(
        "bf16", x, r, w, 1e-6, None, dynamic=True)
    assert g1 == g2 and np.array_equal(p1, p2) and np.array_equal(y1, y2)
    assert np.array_equal(sf2, O.nvfp4_swizzle_scales(sf1.reshape(rows, hidden // 16), hidden))


def test_large_nvfp4_16384x7168_swizzled_matches_linear():
    rows, hidden = 16384, 7168
    x, r, w = synth.rows_input(0, rows, hidden, "bf16", outlier_frac=0.01)
    gs = oracle_gs("bf16", x, r, w, 1e-6)
    (s1, y1, p1, sf1, _), (s2, y2, p2, sf2, _) = run_linear_and_swizzled("bf16", x, r, w, 1e-6, gs)
    assert np.array_equal(p1, p2) and np.array_equal(y1, y2)
    assert np.array_equal(sf2, O.nvfp4_swizzle_scales(sf1.reshape(rows, hidden // 16), hidden))


@pytest.mark.parametrize("rows,hidden", [(512, 7168), (200, 1056)])
def test_kernel_output_feeds_the_block_scaled_gemm(rows, hidden):
    x, r, w = synth.rows_input(7, rows, hidden, "bf16", outlier_frac=0.01)
    gs = oracle_gs("bf16", x, r, w, 1e-6)
    (_, _, p1, sf1, _), (_, _, p2, sf2, _) = run_linear_and_swizzled("bf16", x, r, w, 1e-6, gs)
    pb, sfb = oracle_operand(13, 60, 144, hidden)
    c = gemm_nvfp4(p2, sf2, pb, O.nvfp4_swizzle_scales(sfb, hidden))
    ok, worst = gemm_matches(c, raw_values(p1, sf1.reshape(rows, hidden // 16)), raw_values(pb, sfb))
    assert ok, "GEMM on the kernel's swizzled output is off by %.3g of sum |a b|" % worst
