"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws numbers and stores them in the tensors' storage types.
It holds none of the norm / quantisation arithmetic.  Rounding to bfloat16 and
float16 uses numpy's and torch's own conversions (float64 -> float32 in numpy,
then float32 -> bf16 in torch / float32 -> fp16 in numpy), which gives the same
bytes on x86-64 and aarch64.

Generator: a counter-based splitmix64.  The stream key of (seed, tensor_id) is
mix64(seed * 2^40 + tensor_id); element i draws mix64(key + (i + 1) * gamma)
with gamma = 0x9E3779B97F4A7C15 (the splitmix64 increment).  A uniform in
(0, 1] is ((z >> 11) + 1) * 2^-53, and a standard normal uses the Box-Muller
cosine branch on the uniforms (u[2i], u[2i+1]).

Tensor ids: x = 1, residual = 2, weight = 3, q = 4, k = 5, q weight = 6,
k weight = 7, outlier mask = 8.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 20

TID_X, TID_RES, TID_W, TID_Q, TID_K, TID_QW, TID_KW, TID_OUTLIER = 1, 2, 3, 4, 5, 6, 7, 8


def _mix64(z):
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed, tensor_id):
    with np.errstate(over="ignore"):
        base = np.uint64(seed) * np.uint64(1 << 40) + np.uint64(tensor_id)
    return _mix64(np.array([base], np.uint64))[0]


def _uniform_chunk(key, start, n):
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = _mix64(key + idx * GAMMA)
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def _parallel(n, fn):
    """Run fn(c0, c1) over chunks of [0, n) on a thread pool (numpy releases
    the GIL inside its array loops); chunk results do not depend on the pool."""
    chunks = [(c0, min(n, c0 + _CHUNK)) for c0 in range(0, n, _CHUNK)]
    if len(chunks) <= 1:
        for c in chunks:
            fn(*c)
        return
    workers = max(1, min(len(chunks), os.cpu_count() or 1, 32))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(lambda c: fn(*c), chunks))


def uniform(seed, tensor_id, n, start=0):
    """n uniforms in (0, 1] (float64): elements start .. start+n-1 of the stream."""
    key = _key(seed, tensor_id)
    out = np.empty(n, np.float64)

    def fill(c0, c1):
        out[c0:c1] = _uniform_chunk(key, start + c0, c1 - c0)

    _parallel(n, fill)
    return out


def normal(seed, tensor_id, n):
    """n standard normals (float64), Box-Muller on consecutive uniform pairs."""
    key = _key(seed, tensor_id)
    out = np.empty(n, np.float64)

    def fill(c0, c1):
        u = _uniform_chunk(key, 2 * c0, 2 * (c1 - c0))
        out[c0:c1] = np.sqrt(-2.0 * np.log(u[0::2])) * np.cos(2.0 * np.pi * u[1::2])

    _parallel(n, fill)
    return out


def to_bits(v, dtype):
    """float64 array -> uint16 bit patterns of `dtype` ('bf16' or 'fp16')."""
    f32 = np.ascontiguousarray(v, dtype=np.float64).astype(np.float32)
    if dtype == "bf16":
        t = torch.from_numpy(f32).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    if dtype == "fp16":
        return f32.astype(np.float16).view(np.uint16)
    raise ValueError("dtype must be 'bf16' or 'fp16'")


def normal_tensor(seed, tensor_id, shape, dtype, mean=0.0, std=1.0):
    n = int(np.prod(shape))
    v = mean + std * normal(seed, tensor_id, n)
    return to_bits(v, dtype).reshape(shape)


def rows_input(seed, rows, hidden, dtype, res_std=1.0, outlier_frac=0.0, outlier_mul=20.0):
    """x, residual and weight of one fused add + RMSNorm call.

    x ~ N(0, 1) (optionally with a Bernoulli(outlier_frac) mask multiplying
    entries by outlier_mul before rounding), residual ~ N(0, res_std^2),
    weight = 1 + 0.1 N(0, 1)."""
    n = rows * hidden
    xv = normal(seed, TID_X, n)
    if outlier_frac > 0.0:
        mask = uniform(seed, TID_OUTLIER, n) < outlier_frac
        xv = np.where(mask, xv * outlier_mul, xv)
    x = to_bits(xv, dtype).reshape(rows, hidden)
    del xv
    r = to_bits(res_std * normal(seed, TID_RES, n), dtype).reshape(rows, hidden)
    w = to_bits(1.0 + 0.1 * normal(seed, TID_W, hidden), dtype)
    return x, r, w


def rope_cos_sin(max_pos, head_dim, theta=1.0e6):
    """[max_pos, head_dim] float32 table: cos in the first half, sin in the second.

    Frequency i (i < head_dim/2) is theta^(-2i/head_dim) and the angle at
    position p is p times it; computed in float64 and rounded once to float32.
    This table is an input of the Q/K call, identical for both sides."""
    half = head_dim // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def qk_input(seed, n_tokens, n_q_heads, n_k_heads, head_dim, dtype, theta=1.0e6):
    """q [T, Hq, D], k [T, Hk, D] ~ N(0, 1); per-tensor head weights
    1 + 0.1 N(0, 1) of shape [D]; positions 0..T-1; the RoPE table."""
    q = normal_tensor(seed, TID_Q, (n_tokens, n_q_heads, head_dim), dtype)
    k = normal_tensor(seed, TID_K, (n_tokens, n_k_heads, head_dim), dtype)
    qw = to_bits(1.0 + 0.1 * normal(seed, TID_QW, head_dim), dtype)
    kw = to_bits(1.0 + 0.1 * normal(seed, TID_KW, head_dim), dtype)
    pos = np.arange(n_tokens, dtype=np.int32)
    cs = rope_cos_sin(n_tokens, head_dim, theta)
    return q, k, qw, kw, pos, cs
