"""The C ABI without a GPU: the library loads, exports every entry point that
include/rq.h declares, and rejects bad arguments with the documented status
before any CUDA call (the pointers below are never dereferenced)."""
import ctypes
import os
import re

import pytest

import nvfp4_quant_gb300 as rq
from nvfp4_quant_gb300 import build as rq_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "rq.h")
OK, NULL, SHAPE, DTYPE, MISAL, ALIAS, UNSUP = 0, 1, 2, 3, 4, 5, 6


@pytest.fixture(scope="module")
def L():
    rq_build.build()
    return rq.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rq_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert "rq_add_rmsnorm_nvfp4" in names and len(names) >= 10
    for n in names:
        assert hasattr(L, n), n
        assert n in rq.SIGNATURES, "binding lacks " + n


def test_binding_constants_match_the_header():
    text = open(HEADER).read()
    for name in ("RQ_MAX_HIDDEN", "RQ_QK_HEAD_DIM", "RQ_QK_MAX_HEADS"):
        m = re.search(r"#define\s+%s\s+(\d+)" % name, text)
        assert m and int(m.group(1)) == getattr(rq, name), name


def test_status_strings_and_sizes(L):
    for code in range(8):
        assert L.rq_status_string(code).decode().startswith(rq.STATUS[code])
    assert rq.rq_nvfp4_packed_bytes(64, 8192) == 64 * 4096
    assert rq.rq_nvfp4_scale_bytes(64, 8192) == 64 * 512
    assert rq.rq_nvfp4_scale_bytes(0, 8192) == 0
    assert L.rq_version() >= 100


# distinct, 16-byte aligned fake addresses far apart
A = {n: 0x10000000 * (i + 1) for i, n in enumerate(
    ["x", "r", "ro", "w", "s", "q", "sf", "y", "amax", "pos", "cs", "qs", "ks", "qo", "ko", "k"])}


def fp8(L, **kw):
    a = dict(x=A["x"], r=A["r"], ro=A["ro"], w=A["w"], eps=1e-6, s=A["s"], q=A["q"], y=A["y"],
             rows=16, hidden=128, dt=0)
    a.update(kw)
    return L.rq_add_rmsnorm_fp8(a["x"], a["r"], a["ro"], a["w"], a["eps"], a["s"], a["q"], a["y"],
                                a["rows"], a["hidden"], a["dt"], None)


def nvfp4(L, **kw):
    a = dict(x=A["x"], r=A["r"], ro=A["ro"], w=A["w"], eps=1e-6, s=A["s"], q=A["q"], sf=A["sf"],
             y=A["y"], rows=16, hidden=128, dt=1)
    a.update(kw)
    return L.rq_add_rmsnorm_nvfp4(a["x"], a["r"], a["ro"], a["w"], a["eps"], a["s"], a["q"], a["sf"],
                                  a["y"], a["rows"], a["hidden"], a["dt"], None)


def nvfp4_swz(L, **kw):
    a = dict(x=A["x"], r=A["r"], ro=A["ro"], w=A["w"], eps=1e-6, s=A["s"], q=A["q"], sf=A["sf"],
             y=A["y"], rows=16, hidden=128, dt=1)
    a.update(kw)
    return L.rq_add_rmsnorm_nvfp4_swizzled(a["x"], a["r"], a["ro"], a["w"], a["eps"], a["s"],
                                           a["q"], a["sf"], a["y"], a["rows"], a["hidden"],
                                           a["dt"], None)


def qk(L, **kw):
    a = dict(q=A["x"], k=A["k"], qst=16 * 128, kst=8 * 128, T=32, hq=16, hk=8, hd=128, qw=A["w"],
             kw=A["r"], eps=1e-6, pos=A["pos"], cs=A["cs"], maxp=4096, qs=A["qs"], ks=A["ks"],
             qo=A["qo"], ko=A["ko"], dt=0)
    a.update(kw)
    return L.rq_qk_rmsnorm_rope_fp8(a["q"], a["k"], a["qst"], a["kst"], a["T"], a["hq"], a["hk"],
                                    a["hd"], a["qw"], a["kw"], a["eps"], a["pos"], a["cs"],
                                    a["maxp"], a["qs"], a["ks"], a["qo"], a["ko"], a["dt"], None)


@pytest.mark.parametrize("call", [fp8, nvfp4, nvfp4_swz])
def test_row_call_rejections(L, call):
    assert call(L, rows=0) == OK  # nothing to do, no launch
    assert call(L, rows=0, x=None, r=None, ro=None, q=None) == OK  # empty tensors, null data
    assert call(L, x=None) == NULL
    assert call(L, w=None) == NULL
    assert call(L, s=None) == NULL
    assert call(L, q=None) == NULL
    assert call(L, rows=-1) == SHAPE
    assert call(L, rows=0, hidden=136) == SHAPE
    assert call(L, rows=0, dt=7) == DTYPE
    assert call(L, hidden=0) == SHAPE
    assert call(L, hidden=136) == SHAPE  # not a multiple of 16
    assert call(L, hidden=rq.RQ_MAX_HIDDEN + 16) == UNSUP
    assert call(L, dt=2) == DTYPE
    assert call(L, x=A["x"] + 8) == MISAL
    assert call(L, q=A["q"] + 4) == MISAL
    assert call(L, y=A["y"] + 2) == MISAL
    assert call(L, s=A["s"] + 2) == MISAL
    # in place residual is allowed, partial overlap is not
    assert call(L, ro=A["r"], rows=0) == OK
    assert call(L, ro=A["r"] + 16) == ALIAS
    assert call(L, ro=A["x"]) == ALIAS
    assert call(L, y=A["ro"]) == ALIAS
    assert call(L, q=A["w"]) == ALIAS
    assert call(L, y=A["s"] - 16) == ALIAS  # norm out covering the scale scalar


def test_nvfp4_specific_rejections(L):
    assert nvfp4(L, sf=None) == NULL
    assert nvfp4(L, sf=A["sf"] + 1) == MISAL
    assert nvfp4(L, sf=A["q"] + 16 * 64 - 16) == ALIAS  # scales inside the packed codes
    assert nvfp4(L, y=None, rows=0) == OK  # norm output is optional


def test_swizzled_scale_size_and_rejections(L):
    # padded to 128-row and 4-block-column multiples
    assert rq.rq_nvfp4_swizzled_scale_bytes(16, 128) == 128 * 8
    assert rq.rq_nvfp4_swizzled_scale_bytes(130, 96) == 256 * 8
    assert rq.rq_nvfp4_swizzled_scale_bytes(128, 64) == 128 * 4
    assert rq.rq_nvfp4_swizzled_scale_bytes(16384, 7168) == 16384 * 448
    assert rq.rq_nvfp4_swizzled_scale_bytes(0, 7168) == 0
    assert nvfp4_swz(L, sf=None) == NULL
    assert nvfp4_swz(L, sf=A["sf"] + 4) == MISAL
    # 16 rows take a whole 128-row tile (1024 bytes here): a scale buffer
    # ending 512 bytes before the packed codes in linear terms overlaps them
    assert nvfp4_swz(L, sf=A["q"] - 512) == ALIAS
    assert nvfp4_swz(L, y=None, rows=0) == OK


def test_gated_rejections(L):
    g = lambda **kw: L.rq_gated_rmsnorm_nvfp4(
        kw.get("x", A["x"]), kw.get("z", A["r"]), kw.get("w", A["w"]), 1e-6, kw.get("s", A["s"]),
        kw.get("q", A["q"]), kw.get("sf", A["sf"]), kw.get("y", A["y"]), kw.get("rows", 16),
        kw.get("hidden", 128), kw.get("dt", 0), None)
    assert g(rows=0, x=None, z=None) == OK
    assert g(z=None) == NULL
    assert g(sf=None) == NULL
    assert g(z=A["r"] + 8) == MISAL
    assert g(hidden=40) == SHAPE
    assert g(dt=3) == DTYPE
    assert g(y=A["r"]) == ALIAS  # nothing may be written over the gate
    assert g(q=A["x"] + 16) == ALIAS
    gz = lambda **kw: L.rq_gated_rmsnorm_nvfp4_swizzled(
        A["x"], A["r"], A["w"], 1e-6, A["s"], A["q"], kw.get("sf", A["sf"]), None, 16, 128, 0, None)
    assert gz(sf=None) == NULL
    assert gz(sf=A["sf"] + 4) == MISAL
    assert gz(sf=A["q"] - 512) == ALIAS  # the padded 1024-byte scale buffer reaches the codes


def test_amax_rejections(L):
    f = lambda **kw: L.rq_add_rmsnorm_amax(kw.get("x", A["x"]), kw.get("r", A["r"]), kw.get("w", A["w"]),
                                           1e-6, kw.get("amax", A["amax"]), kw.get("rows", 4),
                                           kw.get("hidden", 64), kw.get("dt", 0), None)
    assert f(amax=None) == NULL
    assert f(amax=A["amax"] + 2) == MISAL
    assert f(hidden=8) == SHAPE
    assert f(amax=A["x"] + 64) == ALIAS
    assert L.rq_fp8_scale_from_amax(None, A["s"], None) == NULL
    assert L.rq_nvfp4_global_scale_from_amax(A["amax"], A["s"] + 1, None) == MISAL


def test_qk_rejections(L):
    assert qk(L, T=0) == OK
    assert qk(L, T=0, q=None, k=None, pos=None, cs=None) == OK
    assert qk(L, hd=64) == UNSUP
    assert qk(L, dt=5) == DTYPE
    assert qk(L, T=-1) == SHAPE
    assert qk(L, maxp=0) == SHAPE
    assert qk(L, qst=15 * 128) == SHAPE  # stride shorter than the heads of a token
    assert qk(L, qst=16 * 128 + 4) == MISAL
    assert qk(L, pos=None) == NULL
    assert qk(L, cs=None) == NULL
    assert qk(L, qs=None) == NULL
    assert qk(L, k=None) == NULL
    assert qk(L, k=None, kw=None, ks=None, ko=None, hk=0, T=0) == OK  # Q only
    assert qk(L, qo=A["qo"] + 8) == MISAL
    assert qk(L, ko=A["qo"] + 32 * 16 * 128 - 16) == ALIAS
    assert qk(L, qo=A["cs"]) == ALIAS
    # limits that keep byte extents in range
    assert qk(L, maxp=(1 << 40) + 1) == SHAPE
    assert qk(L, qst=(1 << 40) + 8) == SHAPE
    assert qk(L, hq=65537, qst=65537 * 128) == SHAPE


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(rq, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(rq, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        rq.lib()


def test_binding_refuses_host_tensors(L):
    """The Python binding passes device pointers only: a tensor in host
    memory raises before any library call."""
    import torch
    x = torch.zeros((4, 64), dtype=torch.bfloat16)
    w = torch.ones(64, dtype=torch.bfloat16)
    s = torch.ones(1, dtype=torch.float32)
    q = torch.empty((4, 64), dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        rq.rq_add_rmsnorm_fp8(x, x.clone(), torch.empty_like(x), w, 1e-6, s, q)
    with pytest.raises(ValueError, match="CUDA tensor"):
        rq.add_rmsnorm_nvfp4(x, x.clone(), w, 1e-6, s)


def test_dynamic_rejections(L):
    pt = lambda **kw: L.rq_add_rmsnorm_fp8_per_token(
        kw.get("x", A["x"]), kw.get("r", A["r"]), kw.get("ro", A["ro"]), kw.get("w", A["w"]), 1e-6,
        kw.get("q", A["q"]), kw.get("sc", A["s"]), kw.get("y", A["y"]), kw.get("rows", 16),
        kw.get("hidden", 128), 0, None)
    assert pt(rows=0, x=None) == OK
    assert pt(sc=None) == NULL
    assert pt(sc=A["s"] + 2) == MISAL
    assert pt(sc=A["q"] + 64) == ALIAS  # row scales inside the codes
    assert pt(hidden=40) == SHAPE
    dyn = lambda **kw: L.rq_add_rmsnorm_fp8_dynamic(
        kw.get("x", A["x"]), kw.get("r", A["r"]), kw.get("ro", A["ro"]), kw.get("w", A["w"]), 1e-6,
        kw.get("sc", A["s"]), kw.get("q", A["q"]), kw.get("y", None), kw.get("rows", 16), 128, 0,
        None)
    assert dyn(sc=None) == NULL
    assert dyn(sc=A["s"] + 1) == MISAL
    assert dyn(q=None) == NULL
    assert dyn(sc=A["ro"] + 32) == ALIAS
    nv = lambda **kw: L.rq_add_rmsnorm_nvfp4_dynamic(
        A["x"], A["r"], A["ro"], A["w"], 1e-6, kw.get("gs", A["s"]), A["q"], kw.get("sf", A["sf"]),
        None, 16, 128, 1, None)
    assert nv(sf=None) == NULL
    assert nv(sf=A["sf"] + 4) == MISAL
    assert nv(gs=A["sf"]) == ALIAS
    nvs = lambda **kw: L.rq_add_rmsnorm_nvfp4_dynamic_swizzled(
        A["x"], A["r"], A["ro"], A["w"], 1e-6, kw.get("gs", A["s"]), A["q"], kw.get("sf", A["sf"]),
        None, 16, 128, 1, None)
    assert nvs(sf=None) == NULL
    assert nvs(sf=A["sf"] + 4) == MISAL
    assert nvs(gs=A["sf"] + 512) == ALIAS  # inside the padded 1024-byte scale buffer


def test_kv_store_rejections(L):
    f = lambda **kw: L.rq_qk_rmsnorm_rope_fp8_kv_store(
        A["x"], A["k"], 16 * 128, 8 * 128, kw.get("T", 32), 16, kw.get("hk", 8), 128, A["w"], A["r"],
        1e-6, A["pos"], A["cs"], 4096, A["qs"], A["ks"], A["qo"], kw.get("pool", A["ko"]),
        kw.get("slots", A["y"]), kw.get("ns", 100), 0, None)
    assert f(slots=None) == NULL
    assert f(slots=A["y"] + 4) == MISAL
    assert f(ns=-1) == SHAPE
    assert f(pool=A["y"]) == ALIAS  # pool over the slot indices
    assert f(T=0, slots=None) == OK


def test_kv_store_mixed_rejections(L):
    f = lambda **kw: L.rq_qk_rmsnorm_rope_fp8_kv_store_mixed(
        A["x"], A["k"], 16 * 128, 8 * 128, kw.get("T", 32), 16, kw.get("hk", 8), 128,
        kw.get("rd", 64), A["w"], A["r"], 1e-6, A["pos"], A["cs"], 4096, A["qs"], A["ks"], A["qo"],
        kw.get("pool", A["ko"]), kw.get("slots", A["y"]), kw.get("ns", 100), 0, None)
    for rd in (0, 8, 48, 96, 256):
        assert f(rd=rd) == UNSUP
    assert f(slots=None) == NULL
    assert f(slots=A["y"] + 4) == MISAL
    assert f(pool=A["ko"] + 8) == MISAL
    assert f(ns=-1) == SHAPE
    # the pool rows are 8 heads x (128 + 64) bytes: one just below the slot
    # indices reaches into them
    assert f(pool=A["y"] - 100 * 8 * 192 + 16) == ALIAS
    assert f(pool=A["y"] - 100 * 8 * 192) != ALIAS
    assert f(T=0, slots=None) == OK


def test_qk_amax_and_dynamic_rejections(L):
    am = lambda **kw: L.rq_qk_rmsnorm_rope_amax(
        kw.get("q", A["x"]), A["k"], 16 * 128, 8 * 128, 32, 16, kw.get("hk", 8), 128, A["w"],
        A["r"], 1e-6, A["pos"], A["cs"], 4096, kw.get("qa", A["qs"]), kw.get("ka", A["ks"]),
        kw.get("dt", 0), None)
    assert am(qa=None) == NULL
    assert am(ka=None) == NULL
    assert am(qa=A["qs"] + 2) == MISAL
    assert am(qa=A["x"] + 64) == ALIAS  # the maximum inside Q
    assert am(dt=2) == DTYPE
    dyn = lambda **kw: L.rq_qk_rmsnorm_rope_fp8_dynamic(
        A["x"], A["k"], 16 * 128, 8 * 128, 32, 16, 8, 128, A["w"], A["r"], 1e-6, A["pos"], A["cs"],
        4096, kw.get("qs", A["qs"]), kw.get("ks", A["ks"]), kw.get("qo", A["qo"]), A["ko"], 0, None)
    assert dyn(qs=None) == NULL
    assert dyn(ks=A["ks"] + 1) == MISAL
    assert dyn(qs=A["cs"] + 16) == ALIAS
