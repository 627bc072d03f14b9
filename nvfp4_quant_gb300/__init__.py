"""nvfp4_quant_gb300: Python binding of librq, the GB300 (sm_103a) library of
fused residual add + RMSNorm + FP8 / NVFP4 quantisation kernels and the
per-head Q/K RMSNorm + RoPE + FP8 store.

This module only marshals arguments: it turns torch CUDA tensors into device
pointers and sizes, calls the C ABI (include/rq.h) through ctypes, and raises
RQError when a call returns a non-OK status.  Every step of the computation
runs in the CUDA kernels of librq.so; there is no other code path.  If the
library has not been built, importing works but the first call raises.
"""
import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "librq.so")

RQ_BF16, RQ_FP16 = 0, 1
RQ_MAX_HIDDEN = 262144
RQ_QK_HEAD_DIM = 128
RQ_QK_MAX_HEADS = 65536
STATUS = {0: "RQ_OK", 1: "RQ_ERR_NULL", 2: "RQ_ERR_SHAPE", 3: "RQ_ERR_DTYPE",
          4: "RQ_ERR_MISALIGNED", 5: "RQ_ERR_ALIAS", 6: "RQ_ERR_UNSUPPORTED", 7: "RQ_ERR_CUDA"}

# exported symbol -> (restype, argtypes)
_vp, _i64, _f32, _int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
SIGNATURES = {
    "rq_add_rmsnorm_fp8": (_int, [_vp, _vp, _vp, _vp, _f32, _vp, _vp, _vp, _i64, _i64, _int, _vp]),
    "rq_add_rmsnorm_nvfp4": (_int, [_vp, _vp, _vp, _vp, _f32, _vp, _vp, _vp, _vp, _i64, _i64,
                                    _int, _vp]),
    "rq_qk_rmsnorm_rope_fp8": (_int, [_vp, _vp, _i64, _i64, _i64, _int, _int, _int, _vp, _vp,
                                      _f32, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _int, _vp]),
    "rq_qk_rmsnorm_rope_fp8_kv_store": (_int, [_vp, _vp, _i64, _i64, _i64, _int, _int, _int, _vp,
                                               _vp, _f32, _vp, _vp, _i64, _vp, _vp, _vp, _vp,
                                               _vp, _i64, _int, _vp]),
    "rq_qk_rmsnorm_rope_fp8_kv_store_mixed": (_int, [_vp, _vp, _i64, _i64, _i64, _int, _int, _int,
                                                     _int, _vp, _vp, _f32, _vp, _vp, _i64, _vp,
                                                     _vp, _vp, _vp, _vp, _i64, _int, _vp]),
    "rq_qk_rmsnorm_rope_amax": (_int, [_vp, _vp, _i64, _i64, _i64, _int, _int, _int, _vp, _vp,
                                       _f32, _vp, _vp, _i64, _vp, _vp, _int, _vp]),
    "rq_qk_rmsnorm_rope_fp8_dynamic": (_int, [_vp, _vp, _i64, _i64, _i64, _int, _int, _int, _vp,
                                              _vp, _f32, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _int,
                                              _vp]),
    "rq_add_rmsnorm_amax": (_int, [_vp, _vp, _vp, _f32, _vp, _i64, _i64, _int, _vp]),
    "rq_add_rmsnorm_fp8_per_token": (_int, [_vp, _vp, _vp, _vp, _f32, _vp, _vp, _vp, _i64, _i64,
                                            _int, _vp]),
    "rq_add_rmsnorm_fp8_dynamic": (_int, [_vp, _vp, _vp, _vp, _f32, _vp, _vp, _vp, _i64, _i64,
                                          _int, _vp]),
    "rq_add_rmsnorm_nvfp4_dynamic": (_int, [_vp, _vp, _vp, _vp, _f32, _vp, _vp, _vp, _vp, _i64,
                                            _i64, _int, _vp]),
    "rq_fp8_scale_from_amax": (_int, [_vp, _vp, _vp]),
    "rq_nvfp4_global_scale_from_amax": (_int, [_vp, _vp, _vp]),
    "rq_nvfp4_packed_bytes": (ctypes.c_size_t, [_i64, _i64]),
    "rq_nvfp4_scale_bytes": (ctypes.c_size_t, [_i64, _i64]),
    "rq_add_rmsnorm_nvfp4_swizzled": (_int, [_vp, _vp, _vp, _vp, _f32, _vp, _vp, _vp, _vp, _i64,
                                             _i64, _int, _vp]),
    "rq_add_rmsnorm_nvfp4_dynamic_swizzled": (_int, [_vp, _vp, _vp, _vp, _f32, _vp, _vp, _vp, _vp,
                                                     _i64, _i64, _int, _vp]),
    "rq_nvfp4_swizzled_scale_bytes": (ctypes.c_size_t, [_i64, _i64]),
    "rq_gated_rmsnorm_nvfp4": (_int, [_vp, _vp, _vp, _f32, _vp, _vp, _vp, _vp, _i64, _i64, _int,
                                      _vp]),
    "rq_gated_rmsnorm_nvfp4_swizzled": (_int, [_vp, _vp, _vp, _f32, _vp, _vp, _vp, _vp, _i64, _i64,
                                               _int, _vp]),
    "rq_status_string": (ctypes.c_char_p, [_int]),
    "rq_last_error": (ctypes.c_char_p, []),
    "rq_version": (_int, []),
}

_lib = None


class RQError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(message)
        self.status = status


def lib():
    """The loaded librq.so (ctypes); raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("librq.so is not built (%s); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status):
    if status != 0:
        L = lib()
        msg = L.rq_status_string(status).decode()
        if status == 7:
            msg += " (" + L.rq_last_error().decode() + ")"
        raise RQError(status, msg)


def _dt(t):
    if t.dtype == torch.bfloat16:
        return RQ_BF16
    if t.dtype == torch.float16:
        return RQ_FP16
    raise ValueError("tensors must be bfloat16 or float16, got %s" % t.dtype)


def _ptr(t):
    """Device pointer of a CUDA tensor (None for None).  A host tensor is
    refused here: its address would reach the kernels as a device pointer."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("every tensor argument must be a CUDA tensor (got one on %s)" % t.device)
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _out(t, nbytes, name):
    """An output buffer: contiguous, on x's device, and at least nbytes long
    (the kernels write exactly the sizes include/rq.h gives)."""
    if t is None or not t.is_contiguous() or t.numel() * t.element_size() < nbytes:
        raise ValueError("%s must be a contiguous tensor of at least %d bytes" % (name, nbytes))


def _rows(x, *others):
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous [rows, hidden] tensor")
    for o in others:
        if o is not None and (o.shape != x.shape or o.dtype != x.dtype or not o.is_contiguous()):
            raise ValueError("residual / norm_out must match x in shape, dtype and be contiguous")
    return x.shape[0], x.shape[1]


def rq_add_rmsnorm_fp8(x, residual_in, residual_out, weight, eps, scale, q_out,
                       norm_out=None, stream=None):
    """Residual add + RMSNorm + per-tensor FP8 E4M3 (include/rq.h).
    scale: 1-element float32 CUDA tensor (dequant scale); q_out: uint8 [rows, hidden]."""
    rows, hidden = _rows(x, residual_in, residual_out, norm_out)
    if weight.dtype != x.dtype:
        raise ValueError("weight dtype must match x")
    _out(q_out, rows * hidden, "q_out")
    _check(lib().rq_add_rmsnorm_fp8(_ptr(x), _ptr(residual_in), _ptr(residual_out), _ptr(weight),
                                    float(eps), _ptr(scale), _ptr(q_out), _ptr(norm_out),
                                    rows, hidden, _dt(x), _stream(stream)))


def rq_add_rmsnorm_nvfp4(x, residual_in, residual_out, weight, eps, global_scale, q_packed,
                         block_scales, norm_out=None, stream=None):
    """Residual add + RMSNorm (+ norm out) + NVFP4 (include/rq.h).
    q_packed: uint8 [rows, hidden/2]; block_scales: uint8 [rows, hidden/16]."""
    rows, hidden = _rows(x, residual_in, residual_out, norm_out)
    if weight.dtype != x.dtype:
        raise ValueError("weight dtype must match x")
    _out(q_packed, rows * hidden // 2, "q_packed")
    _out(block_scales, rows * (hidden // 16), "block_scales")
    _check(lib().rq_add_rmsnorm_nvfp4(_ptr(x), _ptr(residual_in), _ptr(residual_out),
                                      _ptr(weight), float(eps), _ptr(global_scale),
                                      _ptr(q_packed), _ptr(block_scales), _ptr(norm_out),
                                      rows, hidden, _dt(x), _stream(stream)))


def rq_gated_rmsnorm_nvfp4(x, z, weight, eps, global_scale, q_packed, block_scales,
                           norm_out=None, stream=None):
    """Gated RMSNorm + NVFP4 (include/rq.h): g = dt(x * dt(silu(z))), RMSNorm,
    NVFP4.  q_packed: uint8 [rows, hidden/2]; block_scales: uint8 [rows, hidden/16]."""
    rows, hidden = _rows(x, z, norm_out)
    if weight.dtype != x.dtype:
        raise ValueError("weight dtype must match x")
    _out(q_packed, rows * hidden // 2, "q_packed")
    _out(block_scales, rows * (hidden // 16), "block_scales")
    _check(lib().rq_gated_rmsnorm_nvfp4(_ptr(x), _ptr(z), _ptr(weight), float(eps),
                                        _ptr(global_scale), _ptr(q_packed), _ptr(block_scales),
                                        _ptr(norm_out), rows, hidden, _dt(x), _stream(stream)))


def rq_gated_rmsnorm_nvfp4_swizzled(x, z, weight, eps, global_scale, q_packed, block_scales,
                                    norm_out=None, stream=None):
    """rq_gated_rmsnorm_nvfp4 with swizzled block scales (include/rq.h);
    block_scales: uint8 of rq_nvfp4_swizzled_scale_bytes(rows, hidden) bytes."""
    rows, hidden = _rows(x, z, norm_out)
    if weight.dtype != x.dtype:
        raise ValueError("weight dtype must match x")
    _out(q_packed, rows * hidden // 2, "q_packed")
    _out(block_scales, rq_nvfp4_swizzled_scale_bytes(rows, hidden), "block_scales")
    _check(lib().rq_gated_rmsnorm_nvfp4_swizzled(
        _ptr(x), _ptr(z), _ptr(weight), float(eps), _ptr(global_scale), _ptr(q_packed),
        _ptr(block_scales), _ptr(norm_out), rows, hidden, _dt(x), _stream(stream)))


def rq_add_rmsnorm_amax(x, residual_in, weight, eps, amax_out, stream=None):
    """amax_out[0] = max |RMSNorm(x + residual) * weight| (include/rq.h)."""
    rows, hidden = _rows(x, residual_in)
    _out(amax_out, 4, "amax_out")
    _check(lib().rq_add_rmsnorm_amax(_ptr(x), _ptr(residual_in), _ptr(weight), float(eps),
                                     _ptr(amax_out), rows, hidden, _dt(x), _stream(stream)))


def rq_add_rmsnorm_fp8_per_token(x, residual_in, residual_out, weight, eps, q_out, row_scales,
                                 norm_out=None, stream=None):
    """Residual add + RMSNorm + FP8 with per-row dynamic scales (include/rq.h).
    row_scales: float32 [rows], written."""
    rows, hidden = _rows(x, residual_in, residual_out, norm_out)
    _out(q_out, rows * hidden, "q_out")
    _out(row_scales, rows * 4, "row_scales")
    _check(lib().rq_add_rmsnorm_fp8_per_token(_ptr(x), _ptr(residual_in), _ptr(residual_out),
                                              _ptr(weight), float(eps), _ptr(q_out),
                                              _ptr(row_scales), _ptr(norm_out), rows, hidden,
                                              _dt(x), _stream(stream)))


def rq_add_rmsnorm_fp8_dynamic(x, residual_in, residual_out, weight, eps, scale_out, q_out,
                               norm_out=None, stream=None):
    """Residual add + RMSNorm + FP8 with the per-tensor scale amax/448 computed
    on the device (include/rq.h); scale_out: 1-element float32, written."""
    rows, hidden = _rows(x, residual_in, residual_out, norm_out)
    _out(q_out, rows * hidden, "q_out")
    _out(scale_out, 4, "scale_out")
    _check(lib().rq_add_rmsnorm_fp8_dynamic(_ptr(x), _ptr(residual_in), _ptr(residual_out),
                                            _ptr(weight), float(eps), _ptr(scale_out), _ptr(q_out),
                                            _ptr(norm_out), rows, hidden, _dt(x), _stream(stream)))


def rq_add_rmsnorm_nvfp4_dynamic(x, residual_in, residual_out, weight, eps, global_scale_out,
                                 q_packed, block_scales, norm_out=None, stream=None):
    """Residual add + RMSNorm + NVFP4 with the global scale 2688/amax computed
    on the device (include/rq.h); global_scale_out: 1-element float32, written."""
    rows, hidden = _rows(x, residual_in, residual_out, norm_out)
    _out(q_packed, rows * hidden // 2, "q_packed")
    _out(block_scales, rows * (hidden // 16), "block_scales")
    _out(global_scale_out, 4, "global_scale_out")
    _check(lib().rq_add_rmsnorm_nvfp4_dynamic(_ptr(x), _ptr(residual_in), _ptr(residual_out),
                                              _ptr(weight), float(eps), _ptr(global_scale_out),
                                              _ptr(q_packed), _ptr(block_scales), _ptr(norm_out),
                                              rows, hidden, _dt(x), _stream(stream)))


def rq_add_rmsnorm_nvfp4_swizzled(x, residual_in, residual_out, weight, eps, global_scale,
                                  q_packed, block_scales, norm_out=None, stream=None):
    """rq_add_rmsnorm_nvfp4 with the block scales in the 128 x 4-tile layout a
    block-scaled NVFP4 GEMM reads (include/rq.h); block_scales: uint8 of
    rq_nvfp4_swizzled_scale_bytes(rows, hidden) bytes, every byte written."""
    rows, hidden = _rows(x, residual_in, residual_out, norm_out)
    if weight.dtype != x.dtype:
        raise ValueError("weight dtype must match x")
    _out(q_packed, rows * hidden // 2, "q_packed")
    _out(block_scales, rq_nvfp4_swizzled_scale_bytes(rows, hidden), "block_scales")
    _check(lib().rq_add_rmsnorm_nvfp4_swizzled(_ptr(x), _ptr(residual_in), _ptr(residual_out),
                                               _ptr(weight), float(eps), _ptr(global_scale),
                                               _ptr(q_packed), _ptr(block_scales), _ptr(norm_out),
                                               rows, hidden, _dt(x), _stream(stream)))


def rq_add_rmsnorm_nvfp4_dynamic_swizzled(x, residual_in, residual_out, weight, eps,
                                          global_scale_out, q_packed, block_scales,
                                          norm_out=None, stream=None):
    """rq_add_rmsnorm_nvfp4_dynamic with swizzled block scales (include/rq.h)."""
    rows, hidden = _rows(x, residual_in, residual_out, norm_out)
    _out(q_packed, rows * hidden // 2, "q_packed")
    _out(block_scales, rq_nvfp4_swizzled_scale_bytes(rows, hidden), "block_scales")
    _out(global_scale_out, 4, "global_scale_out")
    _check(lib().rq_add_rmsnorm_nvfp4_dynamic_swizzled(
        _ptr(x), _ptr(residual_in), _ptr(residual_out), _ptr(weight), float(eps),
        _ptr(global_scale_out), _ptr(q_packed), _ptr(block_scales), _ptr(norm_out), rows, hidden,
        _dt(x), _stream(stream)))


def rq_fp8_scale_from_amax(amax, scale_out, stream=None):
    _check(lib().rq_fp8_scale_from_amax(_ptr(amax), _ptr(scale_out), _stream(stream)))


def rq_nvfp4_global_scale_from_amax(amax, gs_out, stream=None):
    _check(lib().rq_nvfp4_global_scale_from_amax(_ptr(amax), _ptr(gs_out), _stream(stream)))


def _heads(t):
    """(n_tokens, n_heads, token_stride) of a [T, H, 128] view with dense heads."""
    if t is None:
        return 0, 0, 0
    if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
        raise ValueError("q / k must be [tokens, heads, head_dim] views with contiguous heads")
    return t.shape[0], t.shape[1], t.stride(0)


def _qk_buffers(ref, hq, hk, positions, cos_sin_cache, q_out, k_out, rope_dim=None, outs=True):
    """Sizes of the Q/K call's side inputs and dense outputs (k_out None: pool;
    outs False: a call without code outputs)."""
    t, d = ref.shape[0], ref.shape[2]
    if t == 0:
        return
    if positions is None or positions.numel() < t:
        raise ValueError("positions must hold one int32 per token")
    cols = d if rope_dim is None else rope_dim
    if cos_sin_cache is None or cos_sin_cache.dim() != 2 or cos_sin_cache.shape[1] != cols:
        raise ValueError("cos_sin_cache must be a [max_pos, %d] float32 tensor" % cols)
    if not outs:
        return
    if hq > 0:
        _out(q_out, t * hq * d, "q_out")
    if hk > 0 and k_out is not None:
        _out(k_out, t * hk * d, "k_out")


def rq_qk_rmsnorm_rope_fp8(q, k, q_weight, k_weight, eps, positions, cos_sin_cache,
                           q_scale, k_scale, q_out, k_out, stream=None):
    """Per-head Q/K RMSNorm + NeoX RoPE + FP8 E4M3 store (include/rq.h).
    q / k may be token-strided views into a fused QKV buffer."""
    tq, hq, sq = _heads(q)
    tk, hk, sk = _heads(k)
    ref = q if q is not None else k
    if q is not None and k is not None and (tq != tk or q.dtype != k.dtype):
        raise ValueError("q and k must have the same token count and dtype")
    head_dim = ref.shape[2]
    _qk_buffers(ref, hq, hk, positions, cos_sin_cache, q_out, k_out)
    _check(lib().rq_qk_rmsnorm_rope_fp8(
        _ptr(q), _ptr(k), sq, sk, ref.shape[0], hq, hk, head_dim, _ptr(q_weight),
        _ptr(k_weight), float(eps), _ptr(positions), _ptr(cos_sin_cache),
        cos_sin_cache.shape[0], _ptr(q_scale), _ptr(k_scale), _ptr(q_out), _ptr(k_out),
        _dt(ref), _stream(stream)))


def rq_qk_rmsnorm_rope_fp8_kv_store(q, k, q_weight, k_weight, eps, positions, cos_sin_cache,
                                    q_scale, k_scale, q_out, k_pool, k_slots, stream=None):
    """Q/K RMSNorm + RoPE + FP8 with K stored into a KV pool (include/rq.h):
    k_pool uint8 [num_slots, n_k_heads, 128]; k_slots int64 [n_tokens]."""
    tq, hq, sq = _heads(q)
    tk, hk, sk = _heads(k)
    ref = q if q is not None else k
    if q is not None and k is not None and (tq != tk or q.dtype != k.dtype):
        raise ValueError("q and k must have the same token count and dtype")
    _qk_buffers(ref, hq, hk, positions, cos_sin_cache, q_out, None)
    if hk > 0 and ref.shape[0] > 0:
        if k_pool is None or k_pool.dim() != 3 or k_pool.shape[1:] != (hk, ref.shape[2]) \
                or not k_pool.is_contiguous():
            raise ValueError("k_pool must be a contiguous [num_slots, n_k_heads, head_dim] tensor")
        if k_slots is None or k_slots.dtype != torch.int64 or k_slots.numel() < ref.shape[0]:
            raise ValueError("k_slots must hold one int64 slot per token")
    _check(lib().rq_qk_rmsnorm_rope_fp8_kv_store(
        _ptr(q), _ptr(k), sq, sk, ref.shape[0], hq, hk, ref.shape[2], _ptr(q_weight),
        _ptr(k_weight), float(eps), _ptr(positions), _ptr(cos_sin_cache), cos_sin_cache.shape[0],
        _ptr(q_scale), _ptr(k_scale), _ptr(q_out), _ptr(k_pool), _ptr(k_slots),
        0 if k_pool is None else k_pool.shape[0], _dt(ref), _stream(stream)))


def _qk_pair(q, k):
    tq, hq, sq = _heads(q)
    tk, hk, sk = _heads(k)
    ref = q if q is not None else k
    if q is not None and k is not None and (tq != tk or q.dtype != k.dtype):
        raise ValueError("q and k must have the same token count and dtype")
    return ref, hq, sq, hk, sk


def rq_qk_rmsnorm_rope_fp8_kv_store_mixed(q, k, q_weight, k_weight, eps, positions,
                                          cos_sin_cache, q_scale, k_scale, q_out, k_pool, k_slots,
                                          rope_dim, stream=None):
    """Q/K RMSNorm + NeoX RoPE on the last rope_dim elements of each head; Q's
    FP8 codes dense, K into a mixed KV pool (include/rq.h): k_pool uint8
    [num_slots, n_k_heads, head_dim + rope_dim] (E4M3 of the first head_dim -
    rope_dim elements, then rope_dim dtype values); cos_sin_cache float32
    [max_pos, rope_dim]; k_slots int64 [n_tokens]."""
    ref, hq, sq, hk, sk = _qk_pair(q, k)
    _qk_buffers(ref, hq, hk, positions, cos_sin_cache, q_out, None, rope_dim)
    if hk > 0 and ref.shape[0] > 0:
        row = ref.shape[2] + rope_dim
        if k_pool is None or k_pool.dim() != 3 or k_pool.shape[1:] != (hk, row) \
                or not k_pool.is_contiguous():
            raise ValueError("k_pool must be a contiguous [num_slots, n_k_heads, %d] tensor" % row)
        if k_slots is None or k_slots.dtype != torch.int64 or k_slots.numel() < ref.shape[0]:
            raise ValueError("k_slots must hold one int64 slot per token")
    _check(lib().rq_qk_rmsnorm_rope_fp8_kv_store_mixed(
        _ptr(q), _ptr(k), sq, sk, ref.shape[0], hq, hk, ref.shape[2], int(rope_dim),
        _ptr(q_weight), _ptr(k_weight), float(eps), _ptr(positions), _ptr(cos_sin_cache),
        cos_sin_cache.shape[0], _ptr(q_scale), _ptr(k_scale), _ptr(q_out), _ptr(k_pool),
        _ptr(k_slots), 0 if k_pool is None else k_pool.shape[0], _dt(ref), _stream(stream)))


def rq_qk_rmsnorm_rope_amax(q, k, q_weight, k_weight, eps, positions, cos_sin_cache, q_amax,
                            k_amax, stream=None):
    """q_amax[0] / k_amax[0] = max |o| over Q / K, o the dtype-rounded output of
    the Q/K RMSNorm + RoPE (include/rq.h); they may be the same tensor."""
    ref, hq, sq, hk, sk = _qk_pair(q, k)
    _qk_buffers(ref, hq, hk, positions, cos_sin_cache, None, None, outs=False)
    if hq > 0:
        _out(q_amax, 4, "q_amax")
    if hk > 0:
        _out(k_amax, 4, "k_amax")
    _check(lib().rq_qk_rmsnorm_rope_amax(
        _ptr(q), _ptr(k), sq, sk, ref.shape[0], hq, hk, ref.shape[2], _ptr(q_weight),
        _ptr(k_weight), float(eps), _ptr(positions), _ptr(cos_sin_cache), cos_sin_cache.shape[0],
        _ptr(q_amax), _ptr(k_amax), _dt(ref), _stream(stream)))


def rq_qk_rmsnorm_rope_fp8_dynamic(q, k, q_weight, k_weight, eps, positions, cos_sin_cache,
                                   q_scale_out, k_scale_out, q_out, k_out, stream=None):
    """The Q/K call with per-tensor scales amax(o) / 448 computed on the device
    (include/rq.h); q_scale_out / k_scale_out: 1-element float32, written."""
    ref, hq, sq, hk, sk = _qk_pair(q, k)
    _qk_buffers(ref, hq, hk, positions, cos_sin_cache, q_out, k_out)
    if hq > 0:
        _out(q_scale_out, 4, "q_scale_out")
    if hk > 0:
        _out(k_scale_out, 4, "k_scale_out")
    _check(lib().rq_qk_rmsnorm_rope_fp8_dynamic(
        _ptr(q), _ptr(k), sq, sk, ref.shape[0], hq, hk, ref.shape[2], _ptr(q_weight),
        _ptr(k_weight), float(eps), _ptr(positions), _ptr(cos_sin_cache), cos_sin_cache.shape[0],
        _ptr(q_scale_out), _ptr(k_scale_out), _ptr(q_out), _ptr(k_out), _dt(ref),
        _stream(stream)))


def rq_nvfp4_packed_bytes(rows, hidden):
    return int(lib().rq_nvfp4_packed_bytes(rows, hidden))


def rq_nvfp4_scale_bytes(rows, hidden):
    return int(lib().rq_nvfp4_scale_bytes(rows, hidden))


def rq_nvfp4_swizzled_scale_bytes(rows, hidden):
    return int(lib().rq_nvfp4_swizzled_scale_bytes(rows, hidden))


# ---------------------------------------------------------------- conveniences
def _nvfp4_outputs(x, rows, hidden, swizzled):
    q = torch.empty((rows, hidden // 2), dtype=torch.uint8, device=x.device)
    if swizzled:
        sf = torch.empty((rq_nvfp4_swizzled_scale_bytes(rows, hidden),), dtype=torch.uint8,
                         device=x.device)
    else:
        sf = torch.empty((rows, hidden // 16), dtype=torch.uint8, device=x.device)
    return q, sf


def add_rmsnorm_nvfp4(x, residual, weight, eps, global_scale, with_norm_out=False,
                      in_place=True, swizzled=False, stream=None):
    """Allocate the outputs (torch) and run rq_add_rmsnorm_nvfp4 (or, with
    swizzled, rq_add_rmsnorm_nvfp4_swizzled: block_scales then is the flat
    buffer in the GEMM's tile layout).  Returns (residual_out, q_packed,
    block_scales, norm_out or None)."""
    rows, hidden = _rows(x, residual)
    res_out = residual if in_place else torch.empty_like(x)
    q, sf = _nvfp4_outputs(x, rows, hidden, swizzled)
    y = torch.empty_like(x) if with_norm_out else None
    call = rq_add_rmsnorm_nvfp4_swizzled if swizzled else rq_add_rmsnorm_nvfp4
    call(x, residual, res_out, weight, eps, global_scale, q, sf, y, stream)
    return res_out, q, sf, y


def gated_rmsnorm_nvfp4(x, z, weight, eps, global_scale, with_norm_out=False, swizzled=False,
                        stream=None):
    """Allocate the outputs (torch) and run rq_gated_rmsnorm_nvfp4 (or its
    swizzled form).  Returns (q_packed, block_scales, norm_out or None)."""
    rows, hidden = _rows(x, z)
    q, sf = _nvfp4_outputs(x, rows, hidden, swizzled)
    y = torch.empty_like(x) if with_norm_out else None
    call = rq_gated_rmsnorm_nvfp4_swizzled if swizzled else rq_gated_rmsnorm_nvfp4
    call(x, z, weight, eps, global_scale, q, sf, y, stream)
    return q, sf, y


def qk_rmsnorm_rope_fp8(q, k, q_weight, k_weight, eps, positions, cos_sin_cache, q_scale,
                        k_scale, stream=None):
    """Allocate dense FP8 outputs (torch) and run rq_qk_rmsnorm_rope_fp8.
    Returns (q_out [T, Hq, 128], k_out [T, Hk, 128]); either is None when its
    input is None."""
    q_out = None if q is None else torch.empty(tuple(q.shape), dtype=torch.uint8, device=q.device)
    k_out = None if k is None else torch.empty(tuple(k.shape), dtype=torch.uint8, device=k.device)
    rq_qk_rmsnorm_rope_fp8(q, k, q_weight, k_weight, eps, positions, cos_sin_cache, q_scale,
                           k_scale, q_out, k_out, stream)
    return q_out, k_out


def add_rmsnorm_fp8(x, residual, weight, eps, scale, with_norm_out=False, in_place=True,
                    stream=None):
    """Allocate the outputs (torch) and run rq_add_rmsnorm_fp8.  Returns
    (residual_out, q, norm_out or None)."""
    rows, hidden = _rows(x, residual)
    res_out = residual if in_place else torch.empty_like(x)
    q = torch.empty((rows, hidden), dtype=torch.uint8, device=x.device)
    y = torch.empty_like(x) if with_norm_out else None
    rq_add_rmsnorm_fp8(x, residual, res_out, weight, eps, scale, q, y, stream)
    return res_out, q, y
