"""GPU parity of the per-head Q/K RMSNorm + NeoX RoPE + FP8 store against the
CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import nvfp4_quant_gb300 as rq
import oracle as O
import synth
from nvfp4_quant_gb300 import build as rq_build
from tests.gpu_util import assert_codes, dev16, f32dev, host8

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    rq_build.build()
    rq.lib()


def run_qk(dt, q_src, k_src, qw, kw, pos, cs, qscale, kscale, eps=1e-6):
    """q_src / k_src: (flat uint16 array, n_heads, token_stride) or None."""
    T = len(pos)
    args = {}
    outs = {}
    for name, src in (("q", q_src), ("k", k_src)):
        if src is None:
            args[name] = None
            outs[name] = None
            continue
        flat, heads, stride = src
        buf = dev16(flat, dt)
        view = torch.as_strided(buf, (T, heads, D), (stride, D, 1))
        args[name] = view
        outs[name] = torch.full((T, heads, D), 0xA5, dtype=torch.uint8, device="cuda")
    rq.rq_qk_rmsnorm_rope_fp8(args["q"], args["k"], dev16(qw, dt) if q_src else None,
                              dev16(kw, dt) if k_src else None, eps,
                              torch.from_numpy(np.ascontiguousarray(pos, np.int32)).cuda(),
                              torch.from_numpy(cs).cuda(), f32dev(qscale), f32dev(kscale),
                              outs["q"], outs["k"])
    torch.cuda.synchronize()
    return (host8(outs["q"]) if q_src else None), (host8(outs["k"]) if k_src else None)


def oracle_scales(dt, q, k, qw, kw, pos, cs):
    T, Hq = q.shape[:2]
    Hk = k.shape[1]
    oq = O.qk_rmsnorm_rope(dt, q.reshape(-1), Hq * D, T, Hq, D, qw, 1e-6, pos, cs)
    ok = O.qk_rmsnorm_rope(dt, k.reshape(-1), Hk * D, T, Hk, D, kw, 1e-6, pos, cs)
    return O.fp8_scale_from_amax(O.amax(dt, oq)), O.fp8_scale_from_amax(O.amax(dt, ok))


def check(dt, T, Hq, Hk, seed=0):
    q, k, qw, kw, pos, cs = synth.qk_input(seed, T, Hq, Hk, D, dt)
    qs, ks = oracle_scales(dt, q, k, qw, kw, pos, cs)
    _, qq_ref = O.qk_rmsnorm_rope_fp8(dt, q.reshape(-1), Hq * D, T, Hq, D, qw, 1e-6, pos, cs, qs)
    _, kq_ref = O.qk_rmsnorm_rope_fp8(dt, k.reshape(-1), Hk * D, T, Hk, D, kw, 1e-6, pos, cs, ks)
    qq, kq = run_qk(dt, (q.reshape(-1), Hq, Hq * D), (k.reshape(-1), Hk, Hk * D), qw, kw, pos,
                    cs, qs, ks)
    assert_codes(qq, qq_ref, 0x80, "Q codes")
    assert_codes(kq, kq_ref, 0x80, "K codes")


def test_qk_4096_tokens_16q_8k_heads_bf16():
    check("bf16", 4096, 16, 8)


@pytest.mark.parametrize("T", [1, 2, 3, 33, 1000])
@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_qk_token_counts(T, dt):
    check(dt, T, 5, 3, seed=T)


def test_qk_fused_buffer_strides():
    """Q and K read by token stride out of one [T, 16 + 8 + 8, 128] QKV buffer."""
    T, Hq, Hk, Hv = 257, 16, 8, 8
    q, k, qw, kw, pos, cs = synth.qk_input(3, T, Hq, Hk, D, "bf16")
    fused = np.zeros((T, Hq + Hk + Hv, D), np.uint16)
    fused[:, :Hq] = q
    fused[:, Hq:Hq + Hk] = k
    flat = fused.reshape(-1)
    stride = (Hq + Hk + Hv) * D
    _, qq_ref = O.qk_rmsnorm_rope_fp8("bf16", flat, stride, T, Hq, D, qw, 1e-6, pos, cs, 0.02)
    _, kq_ref = O.qk_rmsnorm_rope_fp8("bf16", flat[Hq * D:], stride, T, Hk, D, kw, 1e-6, pos, cs,
                                      0.03)
    # one device buffer, two strided views
    buf = dev16(flat, "bf16")
    qv = torch.as_strided(buf, (T, Hq, D), (stride, D, 1))
    kv = torch.as_strided(buf, (T, Hk, D), (stride, D, 1), storage_offset=Hq * D)
    qo = torch.empty((T, Hq, D), dtype=torch.uint8, device="cuda")
    ko = torch.empty((T, Hk, D), dtype=torch.uint8, device="cuda")
    rq.rq_qk_rmsnorm_rope_fp8(qv, kv, dev16(qw, "bf16"), dev16(kw, "bf16"), 1e-6,
                              torch.from_numpy(pos).cuda(), torch.from_numpy(cs).cuda(),
                              f32dev(0.02), f32dev(0.03), qo, ko)
    torch.cuda.synchronize()
    assert_codes(host8(qo), qq_ref, 0x80, "Q codes")
    assert_codes(host8(ko), kq_ref, 0x80, "K codes")


def test_qk_q_only_and_clamped_positions():
    T, Hq = 64, 4
    q, k, qw, kw, pos, cs = synth.qk_input(4, T, Hq, 1, D, "bf16")
    bad = pos.copy()
    bad[::5] = -7
    bad[1::7] = 10_000
    clamped = np.clip(bad, 0, T - 1).astype(np.int32)
    _, ref = O.qk_rmsnorm_rope_fp8("bf16", q.reshape(-1), Hq * D, T, Hq, D, qw, 1e-6, clamped, cs,
                                   0.01)
    qq, kq = run_qk("bf16", (q.reshape(-1), Hq, Hq * D), None, qw, kw, bad, cs, 0.01, 1.0)
    assert kq is None
    assert_codes(qq, ref, 0x80, "Q codes")


def test_qk_position_zero_matches_row_norm_kernel():
    """At position 0 RoPE is the identity: the Q/K kernel's codes agree with
    those of the row kernel run on the heads as rows with a zero residual (the
    two sum the squares in different orders, hence the code tolerance)."""
    T, Hq = 128, 8
    q, k, qw, kw, pos, cs = synth.qk_input(5, T, Hq, 1, D, "bf16")
    zero = np.zeros(T, np.int32)
    qq, _ = run_qk("bf16", (q.reshape(-1), Hq, Hq * D), None, qw, kw, zero, cs, 0.01, 1.0)
    x = dev16(q.reshape(T * Hq, D), "bf16")
    r = torch.zeros_like(x)
    codes = torch.empty((T * Hq, D), dtype=torch.uint8, device="cuda")
    rq.rq_add_rmsnorm_fp8(x, r, r, dev16(qw, "bf16"), 1e-6, f32dev(0.01), codes)
    torch.cuda.synchronize()
    assert_codes(qq.reshape(T * Hq, D), host8(codes), 0x80, "Q codes vs row kernel")


@pytest.mark.parametrize("dt", ["bf16", "fp16"])
def test_kv_pool_store(dt):
    """K codes land in pool rows k_slots[t]; slots outside the pool (padding)
    write nothing, other pool rows keep their bytes; Q is dense as usual."""
    T, Hq, Hk, n_slots = 300, 8, 4, 1000
    q, k, qw, kw, pos, cs = synth.qk_input(7, T, Hq, Hk, D, dt)
    rng = np.random.default_rng(7)
    slots = rng.permutation(n_slots)[:T].astype(np.int64)
    slots[::17] = -1
    slots[5] = n_slots + 3  # outside the pool: skipped
    _, qq_ref = O.qk_rmsnorm_rope_fp8(dt, q.reshape(-1), Hq * D, T, Hq, D, qw, 1e-6, pos, cs, 0.02)
    _, kq_ref = O.qk_rmsnorm_rope_fp8(dt, k.reshape(-1), Hk * D, T, Hk, D, kw, 1e-6, pos, cs, 0.03)
    pool_ref = np.full((n_slots, Hk, D), 0x5A, np.uint8)
    ok = (slots >= 0) & (slots < n_slots)
    pool_ref[slots[ok]] = kq_ref[ok]
    pool = torch.full((n_slots, Hk, D), 0x5A, dtype=torch.uint8, device="cuda")
    qo = torch.empty((T, Hq, D), dtype=torch.uint8, device="cuda")
    rq.rq_qk_rmsnorm_rope_fp8_kv_store(dev16(q, dt), dev16(k, dt), dev16(qw, dt), dev16(kw, dt),
                                       1e-6, torch.from_numpy(pos).cuda(),
                                       torch.from_numpy(cs).cuda(), f32dev(0.02), f32dev(0.03),
                                       qo, pool, torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    assert_codes(host8(qo), qq_ref, 0x80, "Q codes")
    got = host8(pool)
    untouched = np.ones(n_slots, bool)
    untouched[slots[ok]] = False
    assert np.all(got[untouched] == 0x5A)
    assert_codes(got[~untouched], pool_ref[~untouched], 0x80, "K pool codes")
