"""Python access to the C oracle (TEST INFRASTRUCTURE ONLY).

Only the tests, the smoke check and the benchmark's CPU-baseline leg import
this package.  The CUDA library and its Python binding never do.

Arrays are numpy: bfloat16/float16 tensors as uint16 bit patterns, E4M3 and
packed E2M1 as uint8.  Each function restates one step of the fused path; the
C source (rq_oracle.c) carries the definitions and the page citations.
"""
import ctypes
import numpy as np

from . import build as _build

BF16, FP16 = 0, 1
_DT = {"bf16": BF16, "fp16": FP16, BF16: BF16, FP16: FP16}

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        dp = ctypes.POINTER(ctypes.c_double)
        fp = ctypes.POINTER(ctypes.c_float)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
        sig = {
            "oracle_bf16_to_double": (ctypes.c_double, [ctypes.c_uint16]),
            "oracle_fp16_to_double": (ctypes.c_double, [ctypes.c_uint16]),
            "oracle_bf16_from_double": (ctypes.c_uint16, [ctypes.c_double]),
            "oracle_fp16_from_double": (ctypes.c_uint16, [ctypes.c_double]),
            "oracle_e4m3_to_double": (ctypes.c_double, [ctypes.c_uint8]),
            "oracle_e4m3_from_double": (ctypes.c_uint8, [ctypes.c_double]),
            "oracle_e2m1_to_double": (ctypes.c_double, [ctypes.c_uint8]),
            "oracle_e2m1_from_double": (ctypes.c_uint8, [ctypes.c_double]),
            "oracle_dt_from_double_array": (None, [i32, dp, i64, u16p]),
            "oracle_dt_to_double_array": (None, [i32, u16p, i64, dp]),
            "oracle_e4m3_from_double_array": (None, [dp, i64, u8p]),
            "oracle_e2m1_from_double_array": (None, [dp, i64, u8p]),
            "oracle_add_rmsnorm": (None, [i32, u16p, u16p, u16p, f32, i64, i64, u16p, u16p]),
            "oracle_quant_fp8": (None, [i32, u16p, i64, f32, u8p]),
            "oracle_quant_nvfp4": (None, [i32, u16p, i64, i64, f32, u8p, u8p]),
            "oracle_add_rmsnorm_fp8": (None, [i32, u16p, u16p, u16p, f32, f32, i64, i64,
                                              u16p, u16p, u8p]),
            "oracle_add_rmsnorm_nvfp4": (None, [i32, u16p, u16p, u16p, f32, f32, i64, i64,
                                                u16p, u16p, u8p, u8p]),
            "oracle_amax": (ctypes.c_float, [i32, u16p, i64]),
            "oracle_nvfp4_swizzled_scale_bytes": (i64, [i64, i64]),
            "oracle_silu_dt": (ctypes.c_uint16, [i32, ctypes.c_uint16]),
            "oracle_gated_rmsnorm": (None, [i32, u16p, u16p, u16p, f32, i64, i64, u16p, u16p]),
            "oracle_gated_rmsnorm_nvfp4": (None, [i32, u16p, u16p, u16p, f32, f32, i64, i64,
                                                  u16p, u16p, u8p, u8p]),
            "oracle_nvfp4_swizzle_scales": (None, [u8p, i64, i64, u8p]),
            "oracle_fp8_scale_from_amax": (ctypes.c_float, [f32]),
            "oracle_fp8_dynamic_scale": (ctypes.c_float, [f32]),
            "oracle_nvfp4_dynamic_gs": (ctypes.c_float, [f32]),
            "oracle_quant_fp8_per_row": (None, [i32, u16p, i64, i64, u8p, fp]),
            "oracle_nvfp4_gs_from_amax": (ctypes.c_float, [f32]),
            "oracle_qk_rmsnorm_rope": (None, [i32, u16p, i64, i64, i32, i32, u16p, f32, i32p,
                                              fp, i64, u16p]),
            "oracle_qk_rmsnorm_rope_fp8": (None, [i32, u16p, i64, i64, i32, i32, u16p, f32,
                                                  i32p, fp, i64, f32, u16p, u8p]),
            "oracle_qk_rmsnorm_rope_partial": (None, [i32, u16p, i64, i64, i32, i32, i32, u16p,
                                                      f32, i32p, fp, i64, u16p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _p(a, ct):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ct))


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


# ---------------------------------------------------------------- formats
def dt_from_double(dt, v):
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint16)
    lib().oracle_dt_from_double_array(_DT[dt], _p(v, ctypes.c_double), v.size,
                                      _p(out, ctypes.c_uint16))
    return out


def dt_to_double(dt, b):
    b = _u16(b)
    out = np.empty(b.shape, np.float64)
    lib().oracle_dt_to_double_array(_DT[dt], _p(b, ctypes.c_uint16), b.size,
                                    _p(out, ctypes.c_double))
    return out


def e4m3_from_double(v):
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint8)
    lib().oracle_e4m3_from_double_array(_p(v, ctypes.c_double), v.size, _p(out, ctypes.c_uint8))
    return out


def e4m3_to_double(c):
    c = np.asarray(c, dtype=np.uint8)
    f = lib().oracle_e4m3_to_double
    return np.array([f(int(x)) for x in c.ravel()], np.float64).reshape(c.shape)


def e2m1_from_double(v):
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, np.uint8)
    lib().oracle_e2m1_from_double_array(_p(v, ctypes.c_double), v.size, _p(out, ctypes.c_uint8))
    return out


def e2m1_to_double(nib):
    nib = np.asarray(nib, dtype=np.uint8)
    f = lib().oracle_e2m1_to_double
    return np.array([f(int(x)) for x in nib.ravel()], np.float64).reshape(nib.shape)


# ---------------------------------------------------------------- fused path
def add_rmsnorm(dt, x, r, w, eps):
    """residual' and the norm output y of a [rows, hidden] call."""
    x, r, w = _u16(x), _u16(r), _u16(w)
    rows, hidden = x.shape
    s = np.empty_like(x)
    y = np.empty_like(x)
    lib().oracle_add_rmsnorm(_DT[dt], _p(x, ctypes.c_uint16), _p(r, ctypes.c_uint16),
                             _p(w, ctypes.c_uint16), eps, rows, hidden,
                             _p(s, ctypes.c_uint16), _p(y, ctypes.c_uint16))
    return s, y


def quant_fp8(dt, y, scale):
    y = _u16(y)
    q = np.empty(y.shape, np.uint8)
    lib().oracle_quant_fp8(_DT[dt], _p(y, ctypes.c_uint16), y.size, scale, _p(q, ctypes.c_uint8))
    return q


def quant_nvfp4(dt, y, gs):
    y = _u16(y)
    rows, hidden = y.shape
    packed = np.empty((rows, hidden // 2), np.uint8)
    sf = np.empty((rows, hidden // 16), np.uint8)
    lib().oracle_quant_nvfp4(_DT[dt], _p(y, ctypes.c_uint16), rows, hidden, gs,
                             _p(packed, ctypes.c_uint8), _p(sf, ctypes.c_uint8))
    return packed, sf


def add_rmsnorm_fp8(dt, x, r, w, eps, scale):
    """(residual', y, q) of the fused FP8 call."""
    x, r, w = _u16(x), _u16(r), _u16(w)
    rows, hidden = x.shape
    s, y = np.empty_like(x), np.empty_like(x)
    q = np.empty(x.shape, np.uint8)
    lib().oracle_add_rmsnorm_fp8(_DT[dt], _p(x, ctypes.c_uint16), _p(r, ctypes.c_uint16),
                                 _p(w, ctypes.c_uint16), eps, scale, rows, hidden,
                                 _p(s, ctypes.c_uint16), _p(y, ctypes.c_uint16),
                                 _p(q, ctypes.c_uint8))
    return s, y, q


def add_rmsnorm_nvfp4(dt, x, r, w, eps, gs):
    """(residual', y, packed codes, block scales) of the fused NVFP4 call."""
    x, r, w = _u16(x), _u16(r), _u16(w)
    rows, hidden = x.shape
    s, y = np.empty_like(x), np.empty_like(x)
    packed = np.empty((rows, hidden // 2), np.uint8)
    sf = np.empty((rows, hidden // 16), np.uint8)
    lib().oracle_add_rmsnorm_nvfp4(_DT[dt], _p(x, ctypes.c_uint16), _p(r, ctypes.c_uint16),
                                   _p(w, ctypes.c_uint16), eps, gs, rows, hidden,
                                   _p(s, ctypes.c_uint16), _p(y, ctypes.c_uint16),
                                   _p(packed, ctypes.c_uint8), _p(sf, ctypes.c_uint8))
    return s, y, packed, sf


def silu_dt(dt, z):
    """dt(silu(z)) for every element of a uint16 array of dtype bits."""
    z = np.asarray(z, np.uint16)
    L = lib()
    return np.fromiter((L.oracle_silu_dt(_DT[dt], int(b)) for b in z.ravel()), np.uint16,
                       count=z.size).reshape(z.shape)


def gated_rmsnorm(dt, x, z, w, eps):
    """(g, y) of the gated RMSNorm: g = dt(x * silu(z)), y = RMSNorm(g) * w."""
    x, z, w = _u16(x), _u16(z), _u16(w)
    rows, hidden = x.shape
    g, y = np.empty_like(x), np.empty_like(x)
    lib().oracle_gated_rmsnorm(_DT[dt], _p(x, ctypes.c_uint16), _p(z, ctypes.c_uint16),
                               _p(w, ctypes.c_uint16), eps, rows, hidden, _p(g, ctypes.c_uint16),
                               _p(y, ctypes.c_uint16))
    return g, y


def gated_rmsnorm_nvfp4(dt, x, z, w, eps, gs):
    """(g, y, packed codes, block scales) of the gated RMSNorm + NVFP4 call."""
    x, z, w = _u16(x), _u16(z), _u16(w)
    rows, hidden = x.shape
    g, y = np.empty_like(x), np.empty_like(x)
    packed = np.empty((rows, hidden // 2), np.uint8)
    sf = np.empty((rows, hidden // 16), np.uint8)
    lib().oracle_gated_rmsnorm_nvfp4(_DT[dt], _p(x, ctypes.c_uint16), _p(z, ctypes.c_uint16),
                                     _p(w, ctypes.c_uint16), eps, gs, rows, hidden,
                                     _p(g, ctypes.c_uint16), _p(y, ctypes.c_uint16),
                                     _p(packed, ctypes.c_uint8), _p(sf, ctypes.c_uint8))
    return g, y, packed, sf


def amax(dt, v):
    v = _u16(v)
    return float(lib().oracle_amax(_DT[dt], _p(v, ctypes.c_uint16), v.size))


def fp8_scale_from_amax(a):
    return float(lib().oracle_fp8_scale_from_amax(a))


def nvfp4_gs_from_amax(a):
    return float(lib().oracle_nvfp4_gs_from_amax(a))


def fp8_dynamic_scale(a):
    return float(lib().oracle_fp8_dynamic_scale(a))


def nvfp4_dynamic_gs(a):
    return float(lib().oracle_nvfp4_dynamic_gs(a))


def quant_fp8_per_row(dt, y):
    """(codes, per-row scales) of the per-token dynamic FP8 quantiser."""
    y = _u16(y)
    rows, hidden = y.shape
    q = np.empty(y.shape, np.uint8)
    sc = np.empty(rows, np.float32)
    lib().oracle_quant_fp8_per_row(_DT[dt], _p(y, ctypes.c_uint16), rows, hidden,
                                   _p(q, ctypes.c_uint8), _p(sc, ctypes.c_float))
    return q, sc


def qk_rmsnorm_rope(dt, src, token_stride, n_tokens, n_heads, head_dim, w, eps,
                    pos, cos_sin):
    """Rounded post-RoPE values o [n_tokens, n_heads, head_dim]; src is a flat
    uint16 array whose token t starts at t*token_stride."""
    src, w = _u16(src), _u16(w)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    cos_sin = np.ascontiguousarray(cos_sin, dtype=np.float32)
    max_pos = cos_sin.shape[0]
    o = np.empty((n_tokens, n_heads, head_dim), np.uint16)
    lib().oracle_qk_rmsnorm_rope(_DT[dt], _p(src, ctypes.c_uint16), token_stride, n_tokens,
                                 n_heads, head_dim, _p(w, ctypes.c_uint16), eps,
                                 _p(pos, ctypes.c_int32), _p(cos_sin, ctypes.c_float),
                                 max_pos, _p(o, ctypes.c_uint16))
    return o


def qk_rmsnorm_rope_fp8(dt, src, token_stride, n_tokens, n_heads, head_dim, w, eps,
                        pos, cos_sin, scale):
    """(o, q) of the fused Q/K call for one of Q or K."""
    src, w = _u16(src), _u16(w)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    cos_sin = np.ascontiguousarray(cos_sin, dtype=np.float32)
    max_pos = cos_sin.shape[0]
    o = np.empty((n_tokens, n_heads, head_dim), np.uint16)
    q = np.empty((n_tokens, n_heads, head_dim), np.uint8)
    lib().oracle_qk_rmsnorm_rope_fp8(_DT[dt], _p(src, ctypes.c_uint16), token_stride,
                                     n_tokens, n_heads, head_dim, _p(w, ctypes.c_uint16),
                                     eps, _p(pos, ctypes.c_int32), _p(cos_sin, ctypes.c_float),
                                     max_pos, scale, _p(o, ctypes.c_uint16),
                                     _p(q, ctypes.c_uint8))
    return o, q


def qk_rmsnorm_rope_partial(dt, src, token_stride, n_tokens, n_heads, head_dim, rope_dim, w,
                            eps, pos, cos_sin):
    """Rounded values o [n_tokens, n_heads, head_dim] with the NeoX rotation on
    the last rope_dim elements of each head only; cos_sin is [max_pos,
    rope_dim]."""
    src, w = _u16(src), _u16(w)
    pos = np.ascontiguousarray(pos, dtype=np.int32)
    cos_sin = np.ascontiguousarray(cos_sin, dtype=np.float32)
    assert cos_sin.shape[1] == rope_dim
    max_pos = cos_sin.shape[0]
    o = np.empty((n_tokens, n_heads, head_dim), np.uint16)
    lib().oracle_qk_rmsnorm_rope_partial(_DT[dt], _p(src, ctypes.c_uint16), token_stride, n_tokens,
                                         n_heads, head_dim, rope_dim, _p(w, ctypes.c_uint16), eps,
                                         _p(pos, ctypes.c_int32), _p(cos_sin, ctypes.c_float),
                                         max_pos, _p(o, ctypes.c_uint16))
    return o


def nvfp4_swizzled_scale_bytes(rows, hidden):
    return int(lib().oracle_nvfp4_swizzled_scale_bytes(rows, hidden))


def nvfp4_swizzle_scales(sf, hidden):
    """Linear [rows, hidden/16] block scales -> the 128 x 4-tile GEMM layout
    (1-D uint8, padding bytes 0)."""
    sf = np.ascontiguousarray(sf, np.uint8)
    rows = sf.shape[0]
    assert sf.shape == (rows, hidden // 16)
    out = np.empty(nvfp4_swizzled_scale_bytes(rows, hidden), np.uint8)
    lib().oracle_nvfp4_swizzle_scales(_p(sf, ctypes.c_uint8), rows, hidden, _p(out, ctypes.c_uint8))
    return out


def nvfp4_dequant(packed, sf, gs):
    """Dequantised values e2m1(c) * sf / gs (float64), shape [rows, hidden]."""
    packed = np.asarray(packed, np.uint8)
    rows = packed.shape[0]
    lo = packed & 0xF
    hi = packed >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(rows, -1)
    e2m1_tab = e2m1_to_double(np.arange(16, dtype=np.uint8))
    e4m3_tab = e4m3_to_double(np.arange(256, dtype=np.uint8))
    vals = e2m1_tab[codes]
    scl = np.repeat(e4m3_tab[np.asarray(sf, np.uint8)], 16, axis=1)
    return vals * scl / gs
