// rq_device.cuh -- device helpers shared by the librq kernels: 128-bit memory
// access with cache hints, dtype packing, FP8/FP4 conversions and group
// reductions.  sm_103a only.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rq {

// ---------------------------------------------------- dependent launches
// Every kernel of the library is launched with programmatic stream
// serialisation allowed, so that its CTAs can be scheduled while the previous
// kernel in the stream drains.  pdl_wait() returns once that kernel has
// finished and its writes are visible; each kernel calls it before its first
// global memory access of any kind.  pdl_trigger() lets the next kernel be
// scheduled as soon as every CTA of this one has called it (it changes when
// the next kernel starts, never what it sees: that kernel waits in turn).
// Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

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
    static __device__ __forceinline__ uint32_t mul2(uint32_t a, uint32_t b)
    {
        uint32_t d;
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
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
    static __device__ __forceinline__ uint32_t mul2(uint32_t a, uint32_t b)
    {
        uint32_t d;
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
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

// ---------------------------------------------------------------- packed fp32
// The product of two fp32 pairs, each half rounded once to nearest even, in a
// form the compiler cannot fuse into a following addition.  Measured on
// GB300: a packed multiply feeding a packed add is contracted into one packed
// FMA (a single rounding) whether written with the __fmul2_rn / __fadd2_rn
// intrinsics or as PTX mul.rn.f32x2 / add.rn.f32x2, and so is an FMA with a
// constant -0 addend.  Here the product is an FMA whose addend nz is -0 known
// only at run time (a kernel argument): RN(a b + -0) = RN(a b), signed zeros
// included, and an FMA result cannot be merged into a later add.
__device__ __forceinline__ float2 mul2_unfused(float2 a, float2 b, float nz)
{
    return __ffma2_rn(a, b, make_float2(nz, nz));
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

// Four fp32 -> four E4M3 bytes in one word, element a in the lowest byte.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d)
{
    uint32_t r;
    asm("{ .reg .b16 lo, hi;\n"
        " cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n"
        " cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n"
        " mov.b32 %0, {lo, hi}; }"
        : "=r"(r) : "f"(a), "f"(b), "f"(c), "f"(d));
    return r;
}

// Eight fp32 -> eight E4M3 bytes, element 0 in the lowest byte of .x.
__device__ __forceinline__ uint2 e4m3x8(const float (&v)[8])
{
    return make_uint2(e4m3x4(v[0], v[1], v[2], v[3]), e4m3x4(v[4], v[5], v[6], v[7]));
}

// The sign bits of 8 dtype values (a 16-byte vector) placed on 8 E4M3 code
// bytes: byte e of the result has bit 7 set where element e is negative.
__device__ __forceinline__ uint2 sign_bytes8(const uint4 &v)
{
    // bytes 1 and 3 of each word hold the sign bits of its two elements at bit 7
    return make_uint2(__byte_perm(v.x, v.y, 0x7531) & 0x80808080u,
                      __byte_perm(v.z, v.w, 0x7531) & 0x80808080u);
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

// |a| / b for two dividends with Blackwell's packed fp32 ops: the steps of
// div_by on |a| without the final copysign (callers put the sign back on the
// encoded result).  Each step is the same IEEE operation on both halves
// (fma(q, -b, m) equals fma(-q, b, m) exactly, negation being exact), so
// every magnitude is bit for bit div_by's.
template <bool kFast>
__device__ __forceinline__ float2 div_mag_by2(float2 a, const Divisor &d)
{
    if (!kFast) return make_float2(div_rn(fabsf(a.x), d.b), div_rn(fabsf(a.y), d.b));
    float2 m;
    asm("{ .reg .f32 t; abs.f32 t, %1; min.NaN.f32 %0, t, %2; }" : "=f"(m.x) : "f"(a.x), "f"(d.clamp));
    asm("{ .reg .f32 t; abs.f32 t, %1; min.NaN.f32 %0, t, %2; }" : "=f"(m.y) : "f"(a.y), "f"(d.clamp));
    const float2 y2 = make_float2(d.y, d.y);
    const float2 q = __fmul2_rn(m, y2);
    const float2 r = __ffma2_rn(q, make_float2(-d.b, -d.b), m);
    return __ffma2_rn(r, y2, q);
}

// ---------------------------------------------------------------- SiLU gate
// The gate of the gated RMSNorm is dt(silu(z)) for a dtype value z, with
// silu(z) = z / (1 + e^-z) rounded once to fp32 and then to the dtype.  It is
// formed exactly: a fast fp32 estimate, a test of whether that estimate lies
// within kSiluUlps fp32 ulps of a point where the dtype rounding changes, and
// a double-precision evaluation for the elements where it does (a small
// fraction of the dtype values; tests/cuda/silu_check.cu checks every one of
// the 65,536 values of each dtype against the oracle's gate).

// Bound on |bits(silu_fast(z)) - bits(RN32(silu(z)))| over every finite fp32
// z >= -87 (the inputs silu_fast is used for): 5, measured over all of them by
// tests/cuda/silu_check.cu.  (The gate's exactness does not rest on it alone:
// the same program checks the final gate of every dtype value.)
constexpr int kSiluUlps = 5;

// silu(z) from u = e^-|z| in (0, 1], which never overflows: sigmoid(z) is
// 1 / (1 + u) for z >= 0 and u / (1 + u) for z < 0, and silu(z) =
// max(z, z * u) / (1 + u) covers both (z * u <= z for z >= 0, >= z for
// z < 0).  u = 2^t * e^d with t = RN(-|z| log2(e)) fed to the ex2.approx
// instruction and d = -|z| - t ln 2, the part of the exponent that rounding t
// dropped, taken in two FMAs with ln 2 split in two parts (the argument
// reduction of Cody and Waite, "Software Manual for the Elementary
// Functions", 1980); e^d is 1 + d to within d^2 / 2 < 2^-37.  The reciprocal
// comes from rcp.approx on [1, 2].  For |z| above about 87, 2^t is below the
// normal range and flushes to zero: silu(z) is then z for z > 0, and the
// caller takes the exact path for z < -87.  |z| is clamped at 128 first, so
// that t and d stay finite for the largest dtype values.
__device__ __forceinline__ float silu_fast(float z)
{
    const float kLog2e = 1.44269502162933349609375f;     // RN(log2 e)
    const float kLn2Hi = 0.693145751953125f;             // ln 2, 16 leading bits
    const float kLn2Lo = 1.42860682030941723212e-6f;     // ln 2 - kLn2Hi
    const float a = fminf(fabsf(z), 128.0f);  // keeps t and d finite for every finite z
    const float t = __fmul_rn(-a, kLog2e);
    float p;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(p) : "f"(t));
    const float d = __fmaf_rn(-t, kLn2Lo, __fmaf_rn(-t, kLn2Hi, -a));
    const float u = __fmaf_rn(p, d, p);
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(__fadd_rn(1.0f, u)));
    return __fmul_rn(fmaxf(z, __fmul_rn(z, u)), r);
}

// ---- double-float arithmetic: a value h + l held as two floats with
// |l| <= ulp(h) / 2.  The error-free sum and product of two floats are
// Dekker's ("A floating-point technique for extending the available
// precision", Numer. Math. 18, 1971; also Knuth, TAOCP vol. 2, 4.2.2), the
// product through one FMA.
struct F2 {
    float h, l;
};

// a + b exactly, for |a| >= |b| (or a == 0)
__device__ __forceinline__ F2 fast_two_sum(float a, float b)
{
    const float s = __fadd_rn(a, b);
    return F2{s, __fsub_rn(b, __fsub_rn(s, a))};
}

// a + b exactly, any order of magnitude
__device__ __forceinline__ F2 two_sum(float a, float b)
{
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    return F2{s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}

// a * b exactly (barring underflow)
__device__ __forceinline__ F2 two_prod(float a, float b)
{
    const float p = __fmul_rn(a, b);
    return F2{p, __fmaf_rn(a, b, -p)};
}

// x * y + c as a double-float, for a float x and double-floats y, c with
// |x y| < |c.h| (the Taylor steps below); error about 2^-46 |c|.
__device__ __forceinline__ F2 df_fma(float x, const F2 &y, const F2 &c)
{
    F2 pr = two_prod(x, y.h);
    pr.l = __fmaf_rn(x, y.l, pr.l);
    const F2 sm = fast_two_sum(c.h, pr.h);
    return fast_two_sum(sm.h, __fadd_rn(__fadd_rn(sm.l, pr.l), c.l));
}

// silu(z) = z / (1 + e^-z) to a relative error of about 2^-43, in fp32
// arithmetic, for -87 <= z <= 87 (the exact path of the gate; the double
// precision units of this GPU run at a small fraction of the fp32 rate):
//   e^-|z| = 2^-k e^-r, k = rint(|z| log2 e), r = |z| - k ln 2 with ln 2 in
//     three parts (Cody and Waite; k ln2_1 and |z| - k ln2_1 are exact);
//   e^s, s = -r, by its Taylor series: the terms of degree 0..7 as
//     double-floats (1/n! as double-floats), grouped in pairs and combined
//     with powers of s (Estrin's scheme, for a short chain of dependent
//     steps), those of degree 8..11, below 2^-26 together, in fp32; the low
//     part of s enters as a factor 1 + s_l;
//   silu = N / D with D = 1 + 2^-k e^s and N = z (z >= 0) or z e^s with the
//     factor 2^-k applied to the quotient (z < 0); the quotient from the
//     reciprocal of D's high part and one correction from the remainder.
// The result is the high part of the double-float quotient: the value
// rounded once to fp32.
__device__ __forceinline__ float silu_df(float z)
{
    if (z == 0.0f) return z;  // silu(+-0) = +-0
    const float kLog2e = 1.44269502162933349609375f;  // RN(log2 e)
    const float kLn2a = 0x1.62e4p-1f;                 // ln 2, 16 leading bits
    const float kLn2b = 0x1.7f7d1cp-20f;              // RN(ln 2 - kLn2a)
    const float kLn2c = 0x1.ef357ap-45f;              // RN(ln 2 - kLn2a - kLn2b)
    const float a = fabsf(z);
    const float k = rintf(__fmul_rn(a, kLog2e));
    // r = a - k ln 2 as a double-float
    const float r1 = __fmaf_rn(-k, kLn2a, a);  // exact
    const F2 kb = two_prod(k, kLn2b);
    F2 r = two_sum(r1, -kb.h);
    r = fast_two_sum(r.h, __fsub_rn(r.l, __fmaf_rn(k, kLn2c, kb.l)));
    const float sh = -r.h, sl = -r.l;  // e^-r = e^(sh + sl), |sh| <= 0.35
    // degrees 8..11 in fp32
    float t = __fmaf_rn(sh, 0x1.ae6456p-26f, 0x1.27e4fcp-22f);  // 1/11!, 1/10!
    t = __fmaf_rn(__fmul_rn(sh, sh), t, __fmaf_rn(sh, 0x1.71de3ap-19f, 0x1.a01a02p-16f));  // 1/9!, 1/8!
    // pairs c_2j + c_2j+1 sh as double-floats
    const F2 p0 = fast_two_sum(1.0f, sh);                                         // 1 + s
    const F2 p1 = df_fma(sh, F2{0x1.555556p-3f, -0x1.555556p-28f}, F2{0.5f, 0.0f});  // 1/2 + s/6
    const F2 p2 = df_fma(sh, F2{0x1.111112p-7f, -0x1.ddddep-32f},
                         F2{0x1.555556p-5f, -0x1.555556p-30f});                  // 1/24 + s/120
    // 1/720 + s/5040 + s^2 t
    const F2 p3 = df_fma(sh, F2{0x1.a01a02p-13f, -0x1.7f97fap-39f},
                         F2{0x1.6c16c2p-10f, __fmaf_rn(__fmul_rn(sh, sh), t, -0x1.27d27ep-35f)});
    // s^2 as a double-float, then (p0 + s2 p1) + s2^2 (p2 + s2 p3)
    const F2 s2 = two_prod(sh, sh);
    auto df_mul_add = [](const F2 &x, const F2 &y, const F2 &c) {  // x * y + c, |x y| < |c|
        F2 pr = two_prod(x.h, y.h);
        pr.l = __fmaf_rn(x.h, y.l, __fmaf_rn(x.l, y.h, pr.l));
        const F2 sm = fast_two_sum(c.h, pr.h);
        return fast_two_sum(sm.h, __fadd_rn(__fadd_rn(sm.l, pr.l), c.l));
    };
    const F2 lo = df_mul_add(s2, p1, p0);
    const F2 hi = df_mul_add(s2, p3, p2);
    F2 s4 = two_prod(s2.h, s2.h);
    s4.l = __fmaf_rn(2.0f * s2.h, s2.l, s4.l);
    F2 acc = df_mul_add(s4, hi, lo);
    // times (1 + sl)
    const F2 e = fast_two_sum(acc.h, __fmaf_rn(acc.h, sl, acc.l));
    // D = 1 + 2^-k e (k <= 126: the scale is a normal power of two)
    const float scale = __int_as_float((127 - (int)k) << 23);
    const float uh = __fmul_rn(e.h, scale), ul = __fmul_rn(e.l, scale);
    const F2 d0 = fast_two_sum(1.0f, uh);
    const F2 d = fast_two_sum(d0.h, __fadd_rn(d0.l, ul));
    // N = z or z e
    F2 nn{z, 0.0f};
    if (z < 0.0f) {
        nn = two_prod(z, e.h);
        nn = fast_two_sum(nn.h, __fmaf_rn(z, e.l, nn.l));
    }
    // Q = N / D: q1 from the reciprocal of d.h, then one correction from the
    // remainder N - q1 D
    float rc;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rc) : "f"(d.h));
    const float q1 = __fmul_rn(nn.h, rc);
    const float rem = __fmaf_rn(-q1, d.l, __fadd_rn(__fmaf_rn(-q1, d.h, nn.h), nn.l));
    const float q = __fadd_rn(q1, __fmul_rn(rem, rc));
    return z < 0.0f ? __fmul_rn(q, scale) : q;
}

// The exact path of the gate: silu(z) rounded once to fp32.  z < -87 (where
// the fp32 result can be subnormal) is evaluated in double precision with
// CUDA's exp.
static __device__ __noinline__ float silu_exact(float z)
{
    if (z < -87.0f) {
        const double zd = z;
        return (float)(zd / (1.0 + exp(-zd)));
    }
    return silu_df(z);
}

// True where the dtype rounding of an fp32 value within kSiluUlps ulps of v
// could differ from that of v, or where silu_fast does not apply (z < -87).
// bf16 keeps the upper 16 bits of the fp32 pattern, so the rounding changes
// where the lower 16 bits pass 0x8000, for normal and subnormal values alike.
// fp16 keeps 10 of the 23 fraction bits for |v| >= 2^-14 (the change at
// 0x1000 of the lower 13 bits); smaller |v| (fp16 subnormals) always take the
// exact path.
template <typename DT>
__device__ __forceinline__ bool silu_near_tie(float v, float z);

template <>
__device__ __forceinline__ bool silu_near_tie<BF16>(float v, float z)
{
    const uint32_t k = (__float_as_uint(v) << 16) + ((uint32_t)(kSiluUlps - 0x8000) << 16);
    return k <= ((uint32_t)(2 * kSiluUlps) << 16) || z < -87.0f;
}

template <>
__device__ __forceinline__ bool silu_near_tie<FP16>(float v, float z)
{
    const uint32_t k = (__float_as_uint(v) << 19) + ((uint32_t)(kSiluUlps - 0x1000) << 19);
    return k <= ((uint32_t)(2 * kSiluUlps) << 19) || fabsf(v) < 0x1p-14f;
}

// The exact gates of the 8 dtype values of one 16-byte vector, as 8 dtype
// values.  `valid` false (a vector past the end of the row, filled with
// zeros) skips the exact path: silu(0) = 0 needs none.
template <typename DT>
__device__ __forceinline__ uint4 silu_gate8(const uint4 &zv, bool valid = true)
{
    float z[8], v[8];
    unpack8<DT>(zv, z);
    uint32_t slow = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        v[e] = silu_fast(z[e]);
        slow |= (uint32_t)silu_near_tie<DT>(v[e], z[e]) << e;
    }
    if (valid && slow != 0) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (slow & (1u << e)) v[e] = silu_exact(z[e]);
    }
    return pack8<DT>(v);
}

// ---------------------------------------------------------------- bf16 gate table
// For bf16 the gated kernel takes its gates from a table in shared memory:
// the exact gates (silu_gate8) of every bf16 value with |z| in [2^-23, 2^9)
// (exponent fields 104 .. 135), both signs, 2 * 4096 entries (16 KB), built
// by each CTA at start (about 1 % of the work of the 16,384 x 7168 call).  A
// vector's gates are then 8 shared-memory loads instead of 8 fast SiLUs and
// their near-tie tests.  The values outside the table have closed forms
// (gate8_bf16).
constexpr uint32_t kGateLo = 104u << 7;  // bf16 pattern of 2^-23
constexpr int kGateHalf = 4096;          // entries per sign

__device__ __forceinline__ void gate_table_fill(uint16_t *tab)
{
    for (int v = threadIdx.x; v < 2 * kGateHalf / 8; v += blockDim.x) {
        const uint32_t e0 = 8u * v;
        const uint32_t b0 = (e0 & (kGateHalf - 1)) + kGateLo + ((e0 & kGateHalf) ? 0x8000u : 0u);
        const uint4 zv = make_uint4(b0 | ((b0 + 1) << 16), (b0 + 2) | ((b0 + 3) << 16),
                                    (b0 + 4) | ((b0 + 5) << 16), (b0 + 6) | ((b0 + 7) << 16));
        sts16(tab + e0, silu_gate8<BF16>(zv));
    }
}

// The exact gates dt(RN32(silu(z))) of 8 bf16 values, from the table where
// all 8 lie in it.  Per 32-bit word (two values), (w & 0x7FFF7FFF) - kGateLo
// in each half is the table index, in range when bits 12..15 of each half are
// clear (a half below the range borrows and sets them; the vector then takes
// the closed forms); the sign bit, moved to bit 12 of its half, selects the
// second half of the table.  Outside the table:
//   |z| < 2^-23:  silu(z) = z/2 + z^2/4 + O(z^4), the second term below
//                 2^-24 |z/2|.  Where z/2 is a bf16 value, every number that
//                 close to it rounds to it; where z/2 is a bf16 midpoint (z
//                 in the lowest binades), z^2/4 is far below fp32's smallest
//                 step, so RN32(silu(z)) is z/2 itself and the dtype rounds
//                 that tie to even.  Either way the gate is dt(z/2), with z/2
//                 exact in fp32 (signed zeros included);
//   |z| >= 512:   e^-|z| < 2^-738: RN32(silu(z)) is z for z > 0 and -0 for
//                 z < 0;
//   inf, NaN:     not defined inputs (+inf gives inf, -inf -0, NaN NaN).
// tests/cuda/silu_check.cu checks this function against the oracle's gate
// for every bf16 value.
__device__ __forceinline__ uint4 gate8_bf16(const uint4 &zv, const uint16_t *tab)
{
    const uint32_t w[4] = {zv.x, zv.y, zv.z, zv.w};
    uint32_t t[4], bad = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t m = (w[k] & 0x7FFF7FFFu) - kGateLo * 0x10001u;
        bad |= m;
        t[k] = m + ((w[k] >> 3) & 0x10001000u);
    }
    uint32_t r[4];
    if ((bad & 0xF000F000u) == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            // plain loads: the table is not written after it is filled, so
            // the compiler may schedule them freely
            r[k] = (uint32_t)tab[t[k] & 0xFFFFu] | ((uint32_t)tab[t[k] >> 16] << 16);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float g[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t b = (w[k] >> (16 * h)) & 0xFFFFu;
                const float z = __uint_as_float(b << 16);
                const uint32_t i = (b & 0x7FFFu) - kGateLo;
                if (i < (uint32_t)kGateHalf) {
                    g[h] = __uint_as_float((uint32_t)tab[i + ((b >> 15) ? kGateHalf : 0)] << 16);
                } else if ((b & 0x7FFFu) < kGateLo) {
                    g[h] = __fmul_rn(z, 0.5f);
                } else {
                    g[h] = z > 0.0f ? z : (z < 0.0f ? -0.0f : z);  // NaN stays NaN
                }
            }
            r[k] = BF16::pack(g[0], g[1]);
        }
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// ---------------------------------------------------------------- fp16 gate table
// The same for fp16, where the table must reach further: it holds the exact
// gates of every fp16 value with |z| < 32 (exponent fields 0 .. 19,
// subnormals included), both signs, 2 * 20,480 entries (80 KB, in dynamic
// shared memory).  Outside it:
//   z >= 32:   e^-z < 2^-46, so z * sigma(z) is within 2^-46 |z| of z and
//              RN32(silu(z)) = z;
//   z <= -32:  |silu(z)| < 32 e^-32 < 2^-41, far below half the smallest fp16
//              subnormal (2^-25): the gate is -0;
//   inf, NaN:  as for bf16.
// tests/cuda/silu_check.cu checks gate8_fp16 against the oracle's gate for
// every fp16 value.
constexpr int kGateHalfF16 = 20 << 10;  // entries per sign

__device__ __forceinline__ void gate_table_fill_fp16(uint16_t *tab)
{
    for (int v = threadIdx.x; v < 2 * kGateHalfF16 / 8; v += blockDim.x) {
        const uint32_t e0 = 8u * v;  // 8 entries, never across the sign boundary
        const uint32_t b0 = e0 < (uint32_t)kGateHalfF16 ? e0 : (e0 - kGateHalfF16) | 0x8000u;
        const uint4 zv = make_uint4(b0 | ((b0 + 1) << 16), (b0 + 2) | ((b0 + 3) << 16),
                                    (b0 + 4) | ((b0 + 5) << 16), (b0 + 6) | ((b0 + 7) << 16));
        sts16(tab + e0, silu_gate8<FP16>(zv));
    }
}

// The exact gates of 8 fp16 values, from the table where all 8 lie in it.
// Per 32-bit word, the magnitude of each half plus its sign times 20,480 is
// the table index (at most 40,959, so no carry between the halves); a half
// with magnitude >= 0x5000 (|z| >= 32) sets bit 15 of magnitude + 0x3000.
__device__ __forceinline__ uint4 gate8_fp16(const uint4 &zv, const uint16_t *tab)
{
    const uint32_t w[4] = {zv.x, zv.y, zv.z, zv.w};
    uint32_t t[4], bad = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t m = w[k] & 0x7FFF7FFFu;
        bad |= m + 0x30003000u;
        t[k] = m + ((w[k] >> 15) & 0x00010001u) * (uint32_t)kGateHalfF16;
    }
    uint32_t r[4];
    if ((bad & 0x80008000u) == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
            r[k] = (uint32_t)tab[t[k] & 0xFFFFu] | ((uint32_t)tab[t[k] >> 16] << 16);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float g[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t b = (w[k] >> (16 * h)) & 0xFFFFu;
                const uint32_t m = b & 0x7FFFu;
                if (m < 0x5000u) {
                    g[h] = FP16::lo(tab[m + ((b >> 15) ? kGateHalfF16 : 0)]);
                } else {
                    const float z = FP16::lo(b);
                    g[h] = z > 0.0f ? z : (z < 0.0f ? -0.0f : z);  // NaN stays NaN
                }
            }
            r[k] = FP16::pack(g[0], g[1]);
        }
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// Elementwise product of two vectors of 8 dtype values, each rounded to
// nearest even in the dtype.  The fp32 product of two bf16 (fp16) values is
// exact, so this is the fp32 product rounded to the dtype.
template <typename DT>
__device__ __forceinline__ uint4 mul8(const uint4 &a, const uint4 &b)
{
    uint4 d;
    d.x = DT::mul2(a.x, b.x);
    d.y = DT::mul2(a.y, b.y);
    d.z = DT::mul2(a.z, b.z);
    d.w = DT::mul2(a.w, b.w);
    return d;
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
