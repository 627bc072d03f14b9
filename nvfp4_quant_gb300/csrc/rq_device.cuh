// rq_device.cuh -- device helpers shared by the librq kernels: 128-bit memory
// access with cache hints, dtype packing, FP8/FP4 conversions and group
// reductions.  sm_103a only.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rq {

// ---------------------------------------------------------------- memory
// Streaming 16-byte load of data read exactly once (x, residual): no L1
// allocation.  Plain (coherent) load, so it is also correct for the residual
// buffer that the same thread overwrites in place afterwards.
__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16-byte load of data shared by many rows (weight, RoPE table): cached.
__device__ __forceinline__ uint4 ld_keep16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float ld_f32(const float *p)
{
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ int ld_s32(const int32_t *p)
{
    int v;
    asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void st16(void *p, uint4 v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__device__ __forceinline__ void st8(void *p, uint32_t lo, uint32_t hi)
{
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" :: "l"(p), "r"(lo), "r"(hi) : "memory");
}

__device__ __forceinline__ void st4(void *p, uint32_t v)
{
    asm volatile("st.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st1(void *p, uint32_t v)
{
    asm volatile("st.global.u8 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------- shared memory
// Asynchronous 16-byte global -> shared copies (cp.async, bypassing L1).  A
// thread that stages data only for itself waits with cp.async.wait_group and
// needs no barrier.
__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    uint32_t a;
    asm("{ .reg .u64 t; cvta.to.shared.u64 t, %1; cvt.u32.u64 %0, t; }" : "=r"(a) : "l"(p));
    return a;
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_addr(smem)), "l"(gmem)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

__device__ __forceinline__ uint4 lds16(const void *smem)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_addr(smem)) : "memory");
    return v;
}

__device__ __forceinline__ void sts16(void *smem, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "r"(smem_addr(smem)), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// ---------------------------------------------------------------- dtypes
// A 32-bit word holds two 16-bit elements, the lower-addressed one in the
// low half.  Unpacking is exact; packing rounds to nearest even.
struct BF16 {
    static __device__ __forceinline__ float lo(uint32_t u) { return __uint_as_float(u << 16); }
    static __device__ __forceinline__ float hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }
    static __device__ __forceinline__ uint32_t pack(float lo_v, float hi_v)
    {
        uint32_t d;
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi_v), "f"(lo_v));
        return d;
    }
};

struct FP16 {
    static __device__ __forceinline__ float lo(uint32_t u)
    {
        float f;
        asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.f32.f16 %0, l; }" : "=f"(f) : "r"(u));
        return f;
    }
    static __device__ __forceinline__ float hi(uint32_t u)
    {
        float f;
        asm("{ .reg .b16 l, h; mov.b32 {l, h}, %1; cvt.f32.f16 %0, h; }" : "=f"(f) : "r"(u));
        return f;
    }
    static __device__ __forceinline__ uint32_t pack(float lo_v, float hi_v)
    {
        uint32_t d;
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi_v), "f"(lo_v));
        return d;
    }
};

// 8 elements of one 16-byte vector as floats
template <typename DT>
__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8])
{
    f[0] = DT::lo(v.x); f[1] = DT::hi(v.x);
    f[2] = DT::lo(v.y); f[3] = DT::hi(v.y);
    f[4] = DT::lo(v.z); f[5] = DT::hi(v.z);
    f[6] = DT::lo(v.w); f[7] = DT::hi(v.w);
}

template <typename DT>
__device__ __forceinline__ uint4 pack8(const float (&f)[8])
{
    uint4 v;
    v.x = DT::pack(f[0], f[1]);
    v.y = DT::pack(f[2], f[3]);
    v.z = DT::pack(f[4], f[5]);
    v.w = DT::pack(f[6], f[7]);
    return v;
}

// ---------------------------------------------------------------- FP8 / FP4
// Two fp32 -> two E4M3 bytes (round to nearest even, satfinite); the first
// argument goes to the lower byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo_v, float hi_v)
{
    uint32_t d;
    asm("{ .reg .b16 t; cvt.rn.satfinite.e4m3x2.f32 t, %1, %2; cvt.u32.u16 %0, t; }"
        : "=r"(d) : "f"(hi_v), "f"(lo_v));
    return d;
}

// Eight fp32 -> eight E4M3 bytes, element 0 in the lowest byte of .x.
__device__ __forceinline__ uint2 e4m3x8(const float (&v)[8])
{
    uint2 r;
    r.x = e4m3x2(v[0], v[1]) | (e4m3x2(v[2], v[3]) << 16);
    r.y = e4m3x2(v[4], v[5]) | (e4m3x2(v[6], v[7]) << 16);
    return r;
}

// Eight fp32 -> eight E2M1 nibbles packed in 32 bits, element 0 in the
// lowest nibble (round to nearest even, satfinite).
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8])
{
    uint32_t d;
    asm("{\n"
        " .reg .b8 b0, b1, b2, b3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
        " mov.b32 %0, {b0, b1, b2, b3};\n"
        "}"
        : "=r"(d)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]),
          "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return d;
}

// Value of an E4M3 byte (exact; the byte comes from e4m3x2, so never NaN).
__device__ __forceinline__ float e4m3_value(uint32_t byte)
{
    float f;
    asm("{ .reg .b16 c; .reg .b32 h2; .reg .b16 lo, hi;\n"
        " cvt.u16.u32 c, %1;\n"
        " cvt.rn.f16x2.e4m3x2 h2, c;\n"
        " mov.b32 {lo, hi}, h2;\n"
        " cvt.f32.f16 %0, lo; }"
        : "=f"(f) : "r"(byte));
    return f;
}

// ---------------------------------------------------------------- division
// IEEE single operations, round to nearest even (PTX rcp.rn / div.rn are the
// correctly rounded reciprocal and quotient).
__device__ __forceinline__ float rcp_rn(float x)
{
    float r;
    asm("rcp.rn.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float div_rn(float a, float b)
{
    float r;
    asm("div.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float mul_rn(float a, float b)
{
    float r;
    asm("mul.rn.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float fma_rn(float a, float b, float c)
{
    float r;
    asm("fma.rn.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// a / b for a divisor b > 0 shared by many dividends (the FP8 dequant scale,
// the constant 6 of the NVFP4 block scale).  Method: Markstein's division
// theorem (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with
// y = RN(1/b) and q = RN(a * y), which is within one ulp of a/b, the remainder
// r = a - b q is exact in one FMA and RN(q + r y) = RN(a/b), barring overflow
// and underflow.  Here it runs on |a| clamped to 2^20 b and the sign of a is
// put back at the end, which makes it branch-free:
//   * for quotients with magnitude in [2^-40, 2^20) the result is the correctly
//     rounded a / b, bit for bit;
//   * larger quotients come out as about 2^20, and quotients below 2^-40 are
//     within one ulp; every consumer here gives those the same code as the true
//     quotient (E4M3 saturates at 448 and rounds anything below 2^-10 to a
//     signed zero);
//   * signed zeros keep their sign, a NaN dividend gives NaN, an infinite one
//     2^20 (E4M3: 448, as satfinite gives for infinity).
// Divisors outside [2^-40, 2^40] (or not positive) must use the IEEE division:
// kernels test Divisor::fast once and run a body instantiated with
// kFast = false for them, so the per-element path has no branch.
struct Divisor {
    float b, y, clamp;
    bool fast;
    __device__ __forceinline__ explicit Divisor(float b_) : b(b_), y(rcp_rn(b_)), clamp(b_ * 0x1p20f)
    {
        fast = b_ >= 0x1p-40f && b_ <= 0x1p40f;
    }
};

template <bool kFast>
__device__ __forceinline__ float div_by(float a, const Divisor &d)
{
    if (!kFast) return div_rn(a, d.b);
    float m;
    asm("{ .reg .f32 t; abs.f32 t, %1; min.NaN.f32 %0, t, %2; }" : "=f"(m) : "f"(a), "f"(d.clamp));
    const float q = mul_rn(m, d.y);
    const float r = fma_rn(-q, d.b, m);
    return copysignf(fma_rn(r, d.y, q), a);
}

// The same division for two dividends with Blackwell's packed fp32 ops: each
// step is the same IEEE operation on both halves (fma(q, -b, m) equals
// fma(-q, b, m) exactly, negation being exact), so every result is bit for
// bit div_by's.
template <bool kFast>
__device__ __forceinline__ float2 div_by2(float2 a, const Divisor &d)
{
    if (!kFast) return make_float2(div_rn(a.x, d.b), div_rn(a.y, d.b));
    float2 m;
    asm("{ .reg .f32 t; abs.f32 t, %1; min.NaN.f32 %0, t, %2; }" : "=f"(m.x) : "f"(a.x), "f"(d.clamp));
    asm("{ .reg .f32 t; abs.f32 t, %1; min.NaN.f32 %0, t, %2; }" : "=f"(m.y) : "f"(a.y), "f"(d.clamp));
    const float2 y2 = make_float2(d.y, d.y);
    const float2 q = __fmul2_rn(m, y2);
    const float2 r = __ffma2_rn(q, make_float2(-d.b, -d.b), m);
    const float2 t = __ffma2_rn(r, y2, q);
    return make_float2(copysignf(t.x, a.x), copysignf(t.y, a.y));
}

// silu(z) = z * sigmoid(z) in fp32.  With u = e^-|z| in (0, 1] (no
// overflow for any z): sigmoid(z) = 1 / (1 + u) for z >= 0 and u / (1 + u)
// for z < 0, the reciprocal from rcp.approx (its argument is in [1, 2]).
// u = 2^t with t = -|z| log2(e) <= 0, split as 2^n * 2^f: n = rint(t), found
// by adding 1.5 * 2^23 (which leaves n in the low bits of the sum), and the
// fraction f = t - n formed with log2(e) in two parts, L1 + L2 (the range
// reduction of Cody and Waite, "Software Manual for the Elementary
// Functions", 1980): f = fma(-|z|, L2, fma(-|z|, L1, -n)), |f| <= 1/2 plus a
// few ulps, so 2^f (in [0.7, 1.42]) comes from the ex2.approx instruction at
// its full relative accuracy whatever |z|.  2^n is applied as 2^(n + 64),
// built in the exponent field, then 2^-64; for z < 0 the product z * 2^f * r
// is formed first and the power of two applied last, so that a result in
// the subnormal range is rounded there once.  t is clamped at -152, below
// which u rounds to 0.  Error against the correctly rounded silu: measured
// over every fp32 input in tests/cuda/silu_check.cu.
__device__ __forceinline__ float silu_f32(float z)
{
    const float kL1 = 1.44269502162933349609375f;  // fp32 nearest log2(e)
    const float kL2 = 1.9259629911266175e-8f;      // log2(e) - kL1
    const float kRound = 12582912.0f;              // 1.5 * 2^23
    const float na = -fabsf(z);
    const float m = __fadd_rn(fmaxf(na * kL1, -152.0f), kRound);
    const float n = __fsub_rn(m, kRound);  // rint(t), exactly
    const float f = __fmaf_rn(na, kL2, __fmaf_rn(na, kL1, -n));
    float p;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(p) : "f"(f));
    // 2^(n + 64): n = bits(m) - bits(1.5 * 2^23), biased by 127
    const float s64 = __int_as_float((__float_as_int(m) - 0x4B400000 + 64 + 127) << 23);
    const float u = __fmul_rn(__fmul_rn(p, s64), 0x1p-64f);
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(__fadd_rn(1.0f, u)));
    const bool pos = z >= 0.0f;  // false for NaN, which stays NaN either way
    const float a = __fmul_rn(__fmul_rn(z, pos ? 1.0f : p), r);
    return __fmul_rn(__fmul_rn(a, pos ? 1.0f : s64), pos ? 1.0f : 0x1p-64f);
}

// ---------------------------------------------------------------- reductions
// Sum over aligned groups of G lanes (G a power of two <= 32) of one warp;
// every lane of the group receives the same result, summed in the same
// order.
template <int G>
__device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

template <int G>
__device__ __forceinline__ float group_max(float v)
{
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

}  // namespace rq
