"""GPU behaviour beyond the numerics: tensors at offsets inside larger
allocations, CUDA-graph capture, concurrent calls from two host threads on
their own streams."""
import threading

import numpy as np
import pytest
import torch

import nvfp4_quant_gb300 as rq
import oracle as O
import synth
from nvfp4_quant_gb300 import build as rq_build
from tests import pins
from tests.gpu_util import assert_codes, dev16, f32dev, host8, host16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    rq_build.build()
    rq.lib()


def test_views_at_aligned_offsets():
    """x, residual and outputs as row slices of larger buffers (16-byte
    aligned, not allocation-aligned) give the same bytes as dense tensors."""
    rows, H = 300, 2048
    x, r, w = synth.rows_input(41, rows, H, "bf16")
    s_ref, y_ref, p_ref, sf_ref = O.add_rmsnorm_nvfp4("bf16", x, r, w, 1e-6, 300.0)
    big_x = torch.zeros((rows + 7, H), dtype=torch.bfloat16, device="cuda")
    big_r = torch.zeros_like(big_x)
    big_x[3:3 + rows] = dev16(x, "bf16")
    big_r[5:5 + rows] = dev16(r, "bf16")
    xv, rv = big_x[3:3 + rows], big_r[5:5 + rows]
    out = torch.zeros((rows + 2, H), dtype=torch.bfloat16, device="cuda")
    yv = out[1:1 + rows]
    pk = torch.zeros((rows + 4, H // 2), dtype=torch.uint8, device="cuda")[2:2 + rows]
    sf = torch.zeros((rows * (H // 16) + 64,), dtype=torch.uint8, device="cuda")[16:16 + rows * (H // 16)]
    rq.rq_add_rmsnorm_nvfp4(xv, rv, rv, dev16(w, "bf16"), 1e-6, f32dev(300.0), pk, sf.view(rows, H // 16), yv)
    torch.cuda.synchronize()
    assert np.array_equal(host16(rv), s_ref)
    p_o, sf_o = O.quant_nvfp4("bf16", host16(yv), 300.0)
    assert np.array_equal(host8(pk), p_o) and np.array_equal(host8(sf).reshape(rows, -1), sf_o)
    assert np.all(host16(big_r[:5]) == 0) and np.all(host16(big_r[5 + rows:]) == 0)


def test_misaligned_view_is_rejected():
    x = torch.zeros((8, 136), dtype=torch.bfloat16, device="cuda")
    v = x.view(-1)[4:4 + 7 * 128].view(7, 128)  # 8-byte offset
    w = torch.ones(128, dtype=torch.bfloat16, device="cuda")
    q = torch.empty((7, 128), dtype=torch.uint8, device="cuda")
    with pytest.raises(rq.RQError) as e:
        rq.rq_add_rmsnorm_fp8(v, v.clone(), torch.empty_like(v.clone()), w, 1e-6, f32dev(1.0), q)
    assert e.value.status == 4


def test_cuda_graph_capture_and_replay():
    """The calls are stream-ordered and allocate nothing, so they can be
    captured; replaying the graph on new inputs gives the eager results."""
    rows, H = 512, 1024
    x1, r1, w = synth.rows_input(42, rows, H, "bf16")
    x2, r2, _ = synth.rows_input(43, rows, H, "bf16")
    xd, rd, wd = dev16(x1, "bf16"), dev16(r1, "bf16"), dev16(w, "bf16")
    ro = torch.empty_like(rd)
    q = torch.empty((rows, H), dtype=torch.uint8, device="cuda")
    sc = f32dev(0.02)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        rq.rq_add_rmsnorm_fp8(xd, rd, ro, wd, 1e-6, sc, q)  # first call: launch set-up
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rq.rq_add_rmsnorm_fp8(xd, rd, ro, wd, 1e-6, sc, q)
    for x, r in ((x1, r1), (x2, r2)):
        xd.copy_(dev16(x, "bf16"))
        rd.copy_(dev16(r, "bf16"))
        g.replay()
        torch.cuda.synchronize()
        s_ref, _, q_ref = O.add_rmsnorm_fp8("bf16", x, r, w, 1e-6, 0.02)
        assert np.array_equal(host16(ro), s_ref)
        assert_codes(host8(q), q_ref, 0x80, "FP8 codes from graph replay")


def test_concurrent_calls_from_two_threads():
    rows, H = 1024, 4096
    inputs = [synth.rows_input(44 + i, rows, H, "fp16") for i in range(2)]
    results = [None, None]

    def work(i):
        torch.cuda.set_device(0)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            x, r, w = (dev16(a, "fp16") for a in inputs[i])
            q = torch.empty((rows, H), dtype=torch.uint8, device="cuda")
            for _ in range(20):
                rq.rq_add_rmsnorm_fp8(x, r, torch.empty_like(r), w, 1e-6, f32dev(0.03), q, stream=s)
            s.synchronize()
            results[i] = host8(q)

    th = [threading.Thread(target=work, args=(i,)) for i in range(2)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    for i in range(2):
        x, r, w = inputs[i]
        _, _, q_ref = O.add_rmsnorm_fp8("fp16", x, r, w, 1e-6, 0.03)
        assert_codes(results[i], q_ref, 0x80, "FP8 codes from thread %d" % i)


def test_every_call_captures_into_one_graph():
    """Every entry point (static, dynamic, per-token, swizzled, gated, Q/K,
    Q/K amax and dynamic, uniform and mixed KV pools) captured in one CUDA
    graph; a replay reproduces the eager outputs bit for bit (the kernels
    are deterministic)."""
    rows, H = 300, 2048
    x, r, w = synth.rows_input(50, rows, H, "bf16")
    xd, rd, wd = dev16(x, "bf16"), dev16(r, "bf16"), dev16(w, "bf16")
    T, Hq, Hk, D = 64, 4, 2, 128
    q, k, qw, kw, pos, cs = synth.qk_input(51, T, Hq, Hk, D, "bf16")
    qd, kd, qwd, kwd = dev16(q, "bf16"), dev16(k, "bf16"), dev16(qw, "bf16"), dev16(kw, "bf16")
    posd, csd = torch.from_numpy(pos).cuda(), torch.from_numpy(cs).cuda()
    u8 = lambda *s: torch.empty(s, dtype=torch.uint8, device="cuda")
    f32 = lambda n: torch.empty(n, dtype=torch.float32, device="cuda")
    out = {"ro": torch.empty_like(rd), "y": torch.empty_like(rd), "q8": u8(rows, H),
           "p": u8(rows, H // 2), "sf": u8(rows, H // 16),
           "sfz": u8(rq.rq_nvfp4_swizzled_scale_bytes(rows, H)), "rs": f32(rows), "s1": f32(1),
           "s2": f32(1), "am": f32(1), "gp": u8(rows, H // 2), "gsf": u8(rows, H // 16),
           "qo": u8(T, Hq, D), "pool": u8(2 * T, Hk, D), "gzp": u8(rows, H // 2),
           "gzs": u8(rq.rq_nvfp4_swizzled_scale_bytes(rows, H)), "qo2": u8(T, Hq, D),
           "ko2": u8(T, Hk, D), "qa": f32(1), "ka": f32(1), "qs": f32(1), "ks": f32(1),
           "qo3": u8(T, Hq, D), "mpool": u8(2 * T, Hk, D + 64)}
    cs64 = torch.from_numpy(synth.rope_cos_sin(T, 64, 1.0e6)).cuda()
    gs, sc = f32dev(300.0), f32dev(0.02)
    slots = torch.randperm(2 * T, generator=torch.Generator().manual_seed(1))[:T].cuda()

    def calls():
        rq.rq_add_rmsnorm_fp8(xd, rd, out["ro"], wd, 1e-6, sc, out["q8"], out["y"])
        rq.rq_add_rmsnorm_nvfp4(xd, rd, out["ro"], wd, 1e-6, gs, out["p"], out["sf"], out["y"])
        rq.rq_add_rmsnorm_nvfp4_dynamic_swizzled(xd, rd, out["ro"], wd, 1e-6, out["s1"], out["p"],
                                                 out["sfz"])
        rq.rq_add_rmsnorm_fp8_per_token(xd, rd, out["ro"], wd, 1e-6, out["q8"], out["rs"])
        rq.rq_add_rmsnorm_fp8_dynamic(xd, rd, out["ro"], wd, 1e-6, out["s2"], out["q8"])
        rq.rq_add_rmsnorm_amax(xd, rd, wd, 1e-6, out["am"])
        rq.rq_gated_rmsnorm_nvfp4(xd, rd, wd, 1e-6, gs, out["gp"], out["gsf"])
        rq.rq_gated_rmsnorm_nvfp4_swizzled(xd, rd, wd, 1e-6, gs, out["gzp"], out["gzs"])
        rq.rq_qk_rmsnorm_rope_fp8_kv_store(qd, kd, qwd, kwd, 1e-6, posd, csd, sc, sc, out["qo"],
                                           out["pool"], slots)
        rq.rq_qk_rmsnorm_rope_amax(qd, kd, qwd, kwd, 1e-6, posd, csd, out["qa"], out["ka"])
        rq.rq_qk_rmsnorm_rope_fp8_dynamic(qd, kd, qwd, kwd, 1e-6, posd, csd, out["qs"], out["ks"],
                                          out["qo2"], out["ko2"])
        rq.rq_qk_rmsnorm_rope_fp8_kv_store_mixed(qd, kd, qwd, kwd, 1e-6, posd, cs64, sc, sc,
                                                 out["qo3"], out["mpool"], slots, 64)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for t in out.values():
            t.zero_()
        calls()  # eager, also the first-call set-up
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in out.items()}
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls()
    for t in out.values():
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    for key in out:
        assert torch.equal(out[key], eager[key]), key


def test_back_to_back_calls_see_each_others_writes():
    """Each kernel may be scheduled while the previous one in the stream
    drains, and waits for it before touching memory.  A chain of in-place
    calls where every call reads the buffer the previous call wrote and
    overwrites the one it read, with no synchronisation between them (eager
    and replayed from a graph), gives the oracle's chain bit for bit; so does
    a Q/K call on codes' inputs that a row call wrote just before it."""
    rows, H, n = 4096, 2048, 6
    a, b, w = synth.rows_input(60, rows, H, "bf16")
    # oracle chain: even calls b <- a + b, odd calls a <- b + a
    ha, hb = a.copy(), b.copy()
    q_ref = []
    for i in range(n):
        x, r = (ha, hb) if i % 2 == 0 else (hb, ha)
        s_ref, _, qr = O.add_rmsnorm_fp8("bf16", x, r, w, 1e-6, 0.05)
        q_ref.append(qr)
        if i % 2 == 0:
            hb = s_ref
        else:
            ha = s_ref
    wd, sc = dev16(w, "bf16"), f32dev(0.05)
    A, B = dev16(a, "bf16"), dev16(b, "bf16")
    qs = [torch.empty((rows, H), dtype=torch.uint8, device="cuda") for _ in range(n)]

    def chain():
        for i in range(n):
            x, r = (A, B) if i % 2 == 0 else (B, A)
            rq.rq_add_rmsnorm_fp8(x, r, r, wd, 1e-6, sc, qs[i])

    def check(tag):
        torch.cuda.synchronize()
        assert np.array_equal(host16(A), ha), tag
        assert np.array_equal(host16(B), hb), tag
        for i in range(n):
            assert_codes(host8(qs[i]), q_ref[i], 0x80, "%s: codes of call %d" % (tag, i))

    chain()
    check("eager")
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g.capture_begin()
        chain()
        g.capture_end()
    torch.cuda.current_stream().wait_stream(s)
    A.copy_(dev16(a, "bf16"))
    B.copy_(dev16(b, "bf16"))
    for t in qs:
        t.zero_()
    g.replay()
    check("graph")

    # a row call writes the Q/K call's Q input in place, the Q/K call reads it
    # right after
    T, Hq, Hk, D = 512, 8, 4, 128
    q, k, qw, kw, pos, cs = synth.qk_input(61, T, Hq, Hk, D, "bf16")
    q2 = q.reshape(T, Hq * D)
    zero = np.zeros_like(q2)
    ones = np.ones(Hq * D, np.float32).view(np.uint32) >> 16  # bf16 1.0
    q_in, _, _ = O.add_rmsnorm_fp8("bf16", q2, zero, ones.astype(np.uint16), 1e-6, 0.05)
    zd = dev16(zero, "bf16")
    q8 = torch.empty((T, Hq * D), dtype=torch.uint8, device="cuda")
    qo, ko = (torch.empty((T, h, D), dtype=torch.uint8, device="cuda") for h in (Hq, Hk))
    rq.rq_add_rmsnorm_fp8(dev16(q2, "bf16"), zd, zd, dev16(ones.astype(np.uint16), "bf16"), 1e-6,
                          sc, q8)
    rq.rq_qk_rmsnorm_rope_fp8(zd.view(T, Hq, D), dev16(k, "bf16"), dev16(qw, "bf16"),
                              dev16(kw, "bf16"), 1e-6, torch.from_numpy(pos).cuda(),
                              torch.from_numpy(cs).cuda(), sc, sc, qo, ko)
    torch.cuda.synchronize()
    _, qq_ref = O.qk_rmsnorm_rope_fp8("bf16", q_in.reshape(-1), Hq * D, T, Hq, D, qw, 1e-6, pos,
                                      cs, 0.05)
    _, kq_ref = O.qk_rmsnorm_rope_fp8("bf16", k.reshape(-1), Hk * D, T, Hk, D, kw, 1e-6, pos, cs,
                                      0.05)
    assert_codes(host8(qo).reshape(qq_ref.shape), qq_ref, 0x80, "Q codes after a row call")
    assert_codes(host8(ko).reshape(kq_ref.shape), kq_ref, 0x80, "K codes after a row call")


def test_calls_around_other_kernels_see_their_writes():
    """A library kernel after a kernel launched without dependent-launch
    attributes (torch's) and before one: the library call reads what torch
    wrote just before it, and torch reads what the library call wrote."""
    rows, H = 2048, 4096
    x, r, w = synth.rows_input(62, rows, H, "fp16")
    xd, rd, wd = dev16(x, "fp16"), dev16(r, "fp16"), dev16(w, "fp16")
    q = torch.empty((rows, H), dtype=torch.uint8, device="cuda")
    sc = f32dev(0.04)
    for _ in range(3):
        rd.mul_(-1.0)  # torch writes the residual (exact: a sign flip)
        rq.rq_add_rmsnorm_fp8(xd, rd, rd, wd, 1e-6, sc, q)  # reads it, writes r' in place
        rd.mul_(0.5)  # torch reads r' right after (exact: a power of two)
    torch.cuda.synchronize()
    hr = r.copy()
    for _ in range(3):
        hr = pins.f64_to_dt(-pins.bits_to_f64(hr, "fp16"), "fp16")
        s_ref, _, q_ref = O.add_rmsnorm_fp8("fp16", x, hr, w, 1e-6, 0.04)
        hr = pins.f64_to_dt(0.5 * pins.bits_to_f64(s_ref, "fp16"), "fp16")
    assert np.array_equal(host16(rd), hr)
    assert_codes(host8(q), q_ref, 0x80, "FP8 codes of the last call")



def test_allocating_conveniences_match_the_explicit_calls():
    """The allocating Python conveniences give the explicit calls' outputs."""
    rows, H = 300, 2048
    x, r, w = synth.rows_input(63, rows, H, "bf16")
    xd, wd = dev16(x, "bf16"), dev16(w, "bf16")
    gs = f32dev(300.0)
    u8 = lambda *s: torch.empty(s, dtype=torch.uint8, device="cuda")
    for swz in (False, True):
        rd = dev16(r, "bf16")
        ro, q, sf, y = rq.add_rmsnorm_nvfp4(xd, rd, wd, 1e-6, gs, with_norm_out=True,
                                            in_place=False, swizzled=swz)
        q2, y2 = u8(rows, H // 2), torch.empty_like(xd)
        sf2 = u8(rq.rq_nvfp4_swizzled_scale_bytes(rows, H)) if swz else u8(rows, H // 16)
        ro2 = torch.empty_like(xd)
        (rq.rq_add_rmsnorm_nvfp4_swizzled if swz else rq.rq_add_rmsnorm_nvfp4)(
            xd, rd, ro2, wd, 1e-6, gs, q2, sf2, y2)
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in ((ro, ro2), (q, q2), (sf, sf2), (y, y2)))
        zd = dev16(r, "bf16")
        q, sf, y = rq.gated_rmsnorm_nvfp4(xd, zd, wd, 1e-6, gs, with_norm_out=True, swizzled=swz)
        (rq.rq_gated_rmsnorm_nvfp4_swizzled if swz else rq.rq_gated_rmsnorm_nvfp4)(
            xd, zd, wd, 1e-6, gs, q2, sf2, y2)
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in ((q, q2), (sf, sf2), (y, y2)))
    T, Hq, Hk, D = 100, 4, 2, 128
    qh, kh, qw, kw, pos, cs = synth.qk_input(64, T, Hq, Hk, D, "bf16")
    args = (dev16(qh, "bf16"), dev16(kh, "bf16"), dev16(qw, "bf16"), dev16(kw, "bf16"), 1e-6,
            torch.from_numpy(pos).cuda(), torch.from_numpy(cs).cuda(), f32dev(0.02), f32dev(0.03))
    qo, ko = rq.qk_rmsnorm_rope_fp8(*args)
    qo2, ko2 = u8(T, Hq, D), u8(T, Hk, D)
    rq.rq_qk_rmsnorm_rope_fp8(*args, qo2, ko2)
    torch.cuda.synchronize()
    assert qo.shape == (T, Hq, D) and torch.equal(qo, qo2) and torch.equal(ko, ko2)
