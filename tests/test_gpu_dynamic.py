"""GPU parity of the dynamic-scale calls (per-token FP8, per-tensor FP8 and
NVFP4 with the scale found on the device) against the CPU oracle."""
import numpy as np
import pytest
import torch

import nvfp4_quant_gb300 as rq
import oracle as O
import synth
from nvfp4_quant_gb300 import build as rq_build
from tests import pins
from tests.gpu_util import (Guarded, assert_codes, assert_norm_within_ulp, assert_nvfp4, dev16,
                            host8, host16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    rq_build.build()
    rq.lib()


def _tdt(dt):
    return torch.bfloat16 if dt == "bf16" else torch.float16


def run_per_token(dt, x, r, w, eps=1e-6):
    rows, H = x.shape
    xd, rd, wd = dev16(x, dt), dev16(r, dt), dev16(w, dt)
    ro, y = Guarded((rows, H), _tdt(dt)), Guarded((rows, H), _tdt(dt))
    q = Guarded((rows, H), torch.uint8)
    sc = Guarded((rows,), torch.float32)
    rq.rq_add_rmsnorm_fp8_per_token(xd, rd, ro.t, wd, eps, q.t, sc.t, y.t)
    torch.cuda.synchronize()
    assert all(g.guards_intact() for g in (ro, y, q, sc))
    return host16(ro.t), host16(y.t), host8(q.t), sc.t.cpu().numpy()


@pytest.mark.parametrize("hidden", [128, 1024, 2064, 7168, 16384])
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_per_token_fp8(hidden, dt):
    rows = max(3, min(600, (1 << 21) // hidden))
    x, r, w = synth.rows_input(31, rows, hidden, dt, outlier_frac=0.01)
    x[1] = 0
    r[1] = 0  # an all-zero row: scale 1, zero codes
    s_ref, y_ref = O.add_rmsnorm(dt, x, r, w, 1e-6)
    q_ref, sc_ref = O.quant_fp8_per_row(dt, y_ref)
    s, y, q, sc = run_per_token(dt, x, r, w)
    assert np.array_equal(s, s_ref)
    assert_norm_within_ulp(y, y_ref, dt)
    assert_codes(q, q_ref, 0x80, "per-token FP8 codes")
    # the quantiser is exact: codes and scales from the kernel's own y
    q_o, sc_o = O.quant_fp8_per_row(dt, y)
    assert np.array_equal(q, q_o) and np.array_equal(sc, sc_o)
    assert sc[1] == 1.0 and np.all(q[1] & 0x7F == 0)
    # a row's scale moves only with its amax (within an ulp of the dtype)
    rel = np.abs(sc.astype(np.float64) / sc_ref - 1.0)
    assert np.all(rel <= 2.0 ** -7)


@pytest.mark.parametrize("hidden", [256, 7168, 40976])
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
@pytest.mark.parametrize("in_place", [False, True])
def test_dynamic_tensor_fp8_and_nvfp4(hidden, dt, in_place):
    rows = 4 * 152 + 3
    x, r, w = synth.rows_input(32, rows, hidden, dt, res_std=2.0, outlier_frac=0.01)
    s_ref, y_ref = O.add_rmsnorm(dt, x, r, w, 1e-6)
    amax = O.amax(dt, y_ref)
    scale_ref, gs_ref = O.fp8_dynamic_scale(amax), O.nvfp4_dynamic_gs(amax)
    q_ref = O.quant_fp8(dt, y_ref, scale_ref)
    p_ref, sf_ref = O.quant_nvfp4(dt, y_ref, gs_ref)

    xd, wd = dev16(x, dt), dev16(w, dt)
    rd = dev16(r, dt)
    ro = rd if in_place else torch.empty_like(rd)
    y = torch.empty_like(xd)
    q = torch.empty((rows, hidden), dtype=torch.uint8, device="cuda")
    sc = torch.full((1,), -5.0, dtype=torch.float32, device="cuda")
    rq.rq_add_rmsnorm_fp8_dynamic(xd, rd, ro, wd, 1e-6, sc, q, y)
    torch.cuda.synchronize()
    assert np.array_equal(host16(ro), s_ref)
    y_gpu = host16(y)
    assert_norm_within_ulp(y_gpu, y_ref, dt)
    s_gpu = float(sc.item())
    assert s_gpu == O.fp8_dynamic_scale(O.amax(dt, y_gpu))
    assert abs(s_gpu / scale_ref - 1.0) <= 2.0 ** -7
    assert np.array_equal(host8(q), O.quant_fp8(dt, y_gpu, s_gpu))
    assert_codes(host8(q), q_ref, 0x80, "dynamic FP8 codes")

    rd = dev16(r, dt)
    ro = rd if in_place else torch.empty_like(rd)
    p = torch.empty((rows, hidden // 2), dtype=torch.uint8, device="cuda")
    sf = torch.empty((rows, hidden // 16), dtype=torch.uint8, device="cuda")
    gs = torch.full((1,), -5.0, dtype=torch.float32, device="cuda")
    rq.rq_add_rmsnorm_nvfp4_dynamic(xd, rd, ro, wd, 1e-6, gs, p, sf, None)
    torch.cuda.synchronize()
    assert np.array_equal(host16(ro), s_ref)
    g_gpu = float(gs.item())
    assert g_gpu == O.nvfp4_dynamic_gs(O.amax(dt, y_gpu))
    p_o, sf_o = O.quant_nvfp4(dt, y_gpu, g_gpu)
    assert np.array_equal(host8(p), p_o) and np.array_equal(host8(sf), sf_o)
    assert_nvfp4(host8(p), host8(sf), p_ref, sf_ref, y_ref, gs_ref, dt)


def test_dynamic_zero_tensor_and_empty():
    x = np.zeros((64, 512), np.uint16)
    _, _, w = synth.rows_input(33, 1, 512, "bf16")
    xd, wd = dev16(x, "bf16"), dev16(w, "bf16")
    rd = torch.zeros_like(xd)
    q = torch.full((64, 512), 0xFF, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(1, dtype=torch.float32, device="cuda")
    rq.rq_add_rmsnorm_fp8_dynamic(xd, rd, rd, wd, 1e-6, sc, q)
    torch.cuda.synchronize()
    assert float(sc.item()) == 1.0 and np.all(host8(q) & 0x7F == 0)
    # no rows: the scale of an empty tensor is 1
    e = torch.zeros((0, 512), dtype=torch.bfloat16, device="cuda")
    sc.fill_(7.0)
    rq.rq_add_rmsnorm_fp8_dynamic(e, e, e, wd, 1e-6, sc, torch.zeros((0, 512), dtype=torch.uint8,
                                                                   device="cuda"))
    torch.cuda.synchronize()
    assert float(sc.item()) == 1.0
