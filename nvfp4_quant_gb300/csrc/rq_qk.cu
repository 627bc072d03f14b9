// rq_qk.cu -- per-head Q/K RMSNorm + NeoX RoPE + uniform FP8 store, and the
// tiny scale-from-amax kernels.
//
// Prior art: "Add NanoJet backend for AutoDeploy prefill-only FP8 inference"
// (TensorRT-LLM PR 17288), Description (fused Q/K RMSNorm and RoPE); "perf:
// add fused norm + RoPE + uniform fp8 store for TRT-LLM DSv4 sparse attention"
// (SGLang PR 32975), review thread (norm + RoPE + uniform FP8 store as one
// kernel epilogue).  The mapping below is ours.
//
// Mapping.  A warp takes one unit of work: 2 * kPairs consecutive heads of one
// token (grid-stride over units, token-major).  A head row (128
// elements = 256 bytes) is owned by 16 lanes, 8 elements (one 16-byte vector)
// per lane: lanes 0-15 take the even heads of the token, lanes 16-31 the odd
// ones.  NeoX RoPE pairs element i with i + 64, i.e. lane l with lane l ^ 8,
// and both lanes of a pair use the same frequencies 8 * (l & 7) .. + 7, so
// each lane loads its 8 cos and 8 sin values once per unit and keeps them in
// registers for all its heads.  The kPairs head loads of a unit are issued
// before any of them is used, so each lane has kPairs 16-byte loads in
// flight; units of a few heads keep the tail of the grid short.  Element
// pairs go through Blackwell's packed fp32 multiply / add / FMA (each half an
// IEEE round-to-nearest operation, so the results are the scalar ones): the
// sum of squares is two interleaved partial sums per lane, then a 16-lane
// shuffle tree; the rounded normalised values are exchanged with one 4-word
// shuffle.
#include "rq_device.cuh"
#include "rq_launch.h"

#include <atomic>

namespace rq {

constexpr int kQKBlock = 128;
constexpr int kHeadDim = 128;
constexpr int kPairs = 4;  // head pairs per step: 8 heads, 4 loads in flight per lane

// QMODE (QKMode): QK_STORE and QK_MIXED write codes; QK_AMAX only reduces
// max |o| per side into *p.q_amax / *p.k_amax (one atomic per CTA each).
// QK_MIXED rotates the last rope_dim = R elements of each head only (lanes
// 16 - R / 8 .. 15; the pair partner of lane l is l ^ (R / 16)) and sends K's
// codes to pool rows of D + R bytes per head: the FP8 codes of the first
// D - R elements, then the last R elements as dtype values.
template <typename DT, bool kFast, int QMODE>
__device__ __forceinline__ void qk_body(const QKParams &p, float (*red)[2])
{
    const int lane16 = threadIdx.x & 15;
    const int half = (threadIdx.x >> 4) & 1;            // even or odd heads
    // rotation geometry: the partner lane (xor), whether this lane holds the
    // upper half of its pairs, the first frequency, and (QK_MIXED) whether
    // the lane's elements are rotated at all
    const int R = QMODE == QK_MIXED ? p.rope_dim : kHeadDim;
    const int xr = R >> 4;
    const bool rotated = QMODE != QK_MIXED || lane16 >= 16 - (R >> 3);
    const bool upper = (lane16 & xr) != 0;
    const int rot = (lane16 & (xr - 1)) * 8;
    const int heads = p.hq + p.hk;
    const int64_t warp0 = ((int64_t)blockIdx.x * kQKBlock + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kQKBlock) >> 5;

    const uint4 qw = p.hq > 0 ? ld_keep16(static_cast<const uint8_t *>(p.qw) + lane16 * 16)
                              : make_uint4(0, 0, 0, 0);
    const uint4 kw = p.hk > 0 ? ld_keep16(static_cast<const uint8_t *>(p.kw) + lane16 * 16)
                              : make_uint4(0, 0, 0, 0);
    const Divisor by_q(QMODE != QK_AMAX && p.hq > 0 ? ld_f32(p.q_scale) : 1.0f);
    const Divisor by_k(QMODE != QK_AMAX && p.hk > 0 ? ld_f32(p.k_scale) : 1.0f);
    float amax_q = 0.0f, amax_k = 0.0f;  // QK_AMAX

    const int groups = (heads + 2 * kPairs - 1) / (2 * kPairs);  // units per token
    // unit = tok * groups + g, stepped by nwarps = step_tok * groups + step_g
    // without a 64-bit division per unit
    const int64_t step_tok = nwarps / groups;
    const int step_g = (int)(nwarps - step_tok * groups);
    int64_t tok = warp0 / groups;
    int g = (int)(warp0 - tok * groups);
    for (; tok < p.n_tokens;) {  // unit < n_units
        const int h0 = g * 2 * kPairs;
        int pos = ld_s32(p.pos + tok);
        pos = pos < 0 ? 0 : (pos >= p.max_pos ? (int)(p.max_pos - 1) : pos);
        const uint8_t *cs = reinterpret_cast<const uint8_t *>(p.cos_sin + (int64_t)pos * R);
        uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0, s0 = c0, s1 = c0;
        if (rotated) {
            c0 = ld_keep16(cs + rot * 4);
            c1 = ld_keep16(cs + rot * 4 + 16);
            s0 = ld_keep16(cs + ((R >> 1) + rot) * 4);
            s1 = ld_keep16(cs + ((R >> 1) + rot) * 4 + 16);
        }
        const float2 cp[4] = {make_float2(__uint_as_float(c0.x), __uint_as_float(c0.y)),
                              make_float2(__uint_as_float(c0.z), __uint_as_float(c0.w)),
                              make_float2(__uint_as_float(c1.x), __uint_as_float(c1.y)),
                              make_float2(__uint_as_float(c1.z), __uint_as_float(c1.w))};
        // lanes holding the lower half of their pairs subtract m * sin, the
        // others add it: fold that sign into the sine once per unit
        // (RN(-x) = -RN(x))
        const uint32_t neg = upper ? 0u : 0x80000000u;
        const float2 sp[4] = {make_float2(__uint_as_float(s0.x ^ neg), __uint_as_float(s0.y ^ neg)),
                              make_float2(__uint_as_float(s0.z ^ neg), __uint_as_float(s0.w ^ neg)),
                              make_float2(__uint_as_float(s1.x ^ neg), __uint_as_float(s1.y ^ neg)),
                              make_float2(__uint_as_float(s1.z ^ neg), __uint_as_float(s1.w ^ neg))};
        const uint8_t *qtok = static_cast<const uint8_t *>(p.q) + tok * p.q_stride * 2;
        const uint8_t *ktok = static_cast<const uint8_t *>(p.k) + tok * p.k_stride * 2;
        // K destination row: the token itself, or its slot in the KV pool
        // (slots outside [0, num_slots) write nothing)
        int64_t krow = tok;
        if (QMODE != QK_AMAX && p.k_slots != nullptr) {
            int64_t sl;
            asm volatile("ld.global.nc.s64 %0, [%1];" : "=l"(sl) : "l"(p.k_slots + tok));
            krow = (sl >= 0 && sl < p.num_slots) ? sl : -1;
        }

        {
            uint4 xv[kPairs];
#pragma unroll
            for (int u = 0; u < kPairs; ++u) {
                const int h = h0 + 2 * u + half;
                const uint8_t *src = h < p.hq ? qtok + (int64_t)h * kHeadDim * 2
                                              : ktok + (int64_t)(h - p.hq) * kHeadDim * 2;
                xv[u] = h < heads ? ld_stream16(src + lane16 * 16) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kPairs; ++u) {
                const int h = h0 + 2 * u + half;
                const bool is_q = h < p.hq;
                // RMSNorm over the 16 lanes of the head row.  Element pairs
                // (2i, 2i+1) go through Blackwell's packed fp32 ops: each half
                // is the same IEEE operation as the scalar one.
                float x[8];
                unpack8<DT>(xv[u], x);
                float2 sq = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 xi = make_float2(x[2 * i], x[2 * i + 1]);
                    sq = __ffma2_rn(xi, xi, sq);  // squares are exact
                }
                const float ss = group_sum<16>(__fadd_rn(sq.x, sq.y));
                // ss / 128 is an exact power-of-two scaling, as the division would
                // be; 1 / sqrt(.) as the correctly rounded reciprocal of the
                // correctly rounded root
                const float rstd =
                    rcp_rn(__fsqrt_rn(__fadd_rn(__fmul_rn(ss, 1.0f / kHeadDim), p.eps)));
                const float2 r2 = make_float2(rstd, rstd);
                float w[8], n[8], m[8];
                unpack8<DT>(is_q ? qw : kw, w);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 ni = __fmul2_rn(__fmul2_rn(make_float2(x[2 * i], x[2 * i + 1]), r2),
                                                 make_float2(w[2 * i], w[2 * i + 1]));
                    n[2 * i] = ni.x;
                    n[2 * i + 1] = ni.y;
                }
                const uint4 nv = pack8<DT>(n);
                // the partner half of each rotation pair
                uint4 pv;
                pv.x = __shfl_xor_sync(0xFFFFFFFFu, nv.x, xr);
                pv.y = __shfl_xor_sync(0xFFFFFFFFu, nv.y, xr);
                pv.z = __shfl_xor_sync(0xFFFFFFFFu, nv.z, xr);
                pv.w = __shfl_xor_sync(0xFFFFFFFFu, nv.w, xr);
                unpack8<DT>(nv, n);
                unpack8<DT>(pv, m);
                float o[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    // two products, each rounded, then their rounded sum (never
                    // one FMA: see mul2_unfused)
                    const float2 oi =
                        __fadd2_rn(mul2_unfused(make_float2(n[2 * i], n[2 * i + 1]), cp[i], p.nz),
                                   mul2_unfused(make_float2(m[2 * i], m[2 * i + 1]), sp[i], p.nz));
                    o[2 * i] = oi.x;
                    o[2 * i + 1] = oi.y;
                }
                uint4 ov = pack8<DT>(o);
                if (QMODE == QK_MIXED && !rotated) ov = nv;  // the unrotated part is n itself
                unpack8<DT>(ov, o);  // FP8 from the dtype-rounded rotation
                if (QMODE == QK_AMAX) {
                    float a = 0.0f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) a = fmaxf(a, fabsf(o[e]));
                    if (h < heads) {
                        if (is_q)
                            amax_q = fmaxf(amax_q, a);
                        else
                            amax_k = fmaxf(amax_k, a);
                    }
                    continue;
                }
                // codes of |o| / scale, then the signs of o on the code bytes
                // (signed zeros included)
                const Divisor &by = is_q ? by_q : by_k;
                float v[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 vi = div_mag_by2<kFast>(make_float2(o[2 * i], o[2 * i + 1]), by);
                    v[2 * i] = vi.x;
                    v[2 * i + 1] = vi.y;
                }
                uint2 code = e4m3x8(v);
                const uint2 sgn = sign_bytes8(ov);
                code.x |= sgn.x;
                code.y |= sgn.y;
                if (h < heads && (is_q || krow >= 0)) {
                    if (QMODE == QK_MIXED && !is_q) {
                        // pool row: D + R bytes per head, codes then dtype values
                        uint8_t *dst = p.k_out + (krow * p.hk + (h - p.hq)) * (int64_t)(kHeadDim + R);
                        const int nope_lanes = 16 - (R >> 3);
                        if (rotated)
                            st16(dst + (kHeadDim - R) + (lane16 - nope_lanes) * 16, ov);
                        else
                            st8(dst + lane16 * 8, code.x, code.y);
                    } else {
                        uint8_t *dst = is_q ? p.q_out + (tok * p.hq + h) * kHeadDim
                                            : p.k_out + (krow * p.hk + (h - p.hq)) * kHeadDim;
                        st8(dst + lane16 * 8, code.x, code.y);
                    }
                }
            }
        }
        tok += step_tok;
        g += step_g;
        if (g >= groups) {
            g -= groups;
            ++tok;
        }
    }

    if (QMODE == QK_AMAX) {
        // block maxima, then one atomic per CTA and side on the float's bits
        // (non-negative floats order like their unsigned bits)
        amax_q = group_max<32>(amax_q);
        amax_k = group_max<32>(amax_k);
        if ((threadIdx.x & 31) == 0) {
            red[threadIdx.x >> 5][0] = amax_q;
            red[threadIdx.x >> 5][1] = amax_k;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            float aq = 0.0f, ak = 0.0f;
            for (int i = 0; i < kQKBlock / 32; ++i) {
                aq = fmaxf(aq, red[i][0]);
                ak = fmaxf(ak, red[i][1]);
            }
            if (p.hq > 0) atomicMax(reinterpret_cast<unsigned int *>(p.q_amax), __float_as_uint(aq));
            if (p.hk > 0) atomicMax(reinterpret_cast<unsigned int *>(p.k_amax), __float_as_uint(ak));
        }
    }
}

template <typename DT, int QMODE>
__global__ void __launch_bounds__(kQKBlock, 6)
qk_rmsnorm_rope_kernel(const QKParams p)
{
    __shared__ float red[kQKBlock / 32][2];
    pdl_trigger();
    pdl_wait();
    const bool fast = QMODE == QK_AMAX || ((p.hq == 0 || Divisor(ld_f32(p.q_scale)).fast) &&
                                          (p.hk == 0 || Divisor(ld_f32(p.k_scale)).fast));
    if (fast)
        qk_body<DT, true, QMODE>(p, red);
    else
        qk_body<DT, false, QMODE>(p, red);
}

template <typename DT, int QMODE>
cudaError_t launch_qk_rmsnorm_rope(const QKParams &p, cudaStream_t stream)
{
    static std::atomic<int> occ_cache[64];
    auto kern = qk_rmsnorm_rope_kernel<DT, QMODE>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int per_sm = dev < 64 ? occ_cache[dev].load(std::memory_order_relaxed) : 0;
    if (per_sm <= 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kQKBlock, 0) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        if (dev < 64) occ_cache[dev].store(per_sm, std::memory_order_relaxed);
    }
    const int groups = (p.hq + p.hk + 2 * kPairs - 1) / (2 * kPairs);
    const int64_t need = (p.n_tokens * groups * 32 + kQKBlock - 1) / kQKBlock;  // a warp per unit
    const int64_t full = (int64_t)device_sms(dev) * per_sm;
    const int grid = (int)(need < full ? need : full);
    return launch_pdl(kern, grid, kQKBlock, 0, stream, p);
}

#define RQ_QK_INSTANTIATE(DT)                                                                      \
    template cudaError_t launch_qk_rmsnorm_rope<DT, QK_STORE>(const QKParams &, cudaStream_t);    \
    template cudaError_t launch_qk_rmsnorm_rope<DT, QK_AMAX>(const QKParams &, cudaStream_t);     \
    template cudaError_t launch_qk_rmsnorm_rope<DT, QK_MIXED>(const QKParams &, cudaStream_t);
RQ_QK_INSTANTIATE(BF16)
RQ_QK_INSTANTIATE(FP16)

// ---- scales from a calibrated amax: one fp32 IEEE division each
__global__ void scale_from_amax_kernel(const float *amax, float *out, int nvfp4, int zero_to_one)
{
    pdl_trigger();
    pdl_wait();
    const float a = *amax;  // plain load: out may alias amax
    *out = (zero_to_one && !(a > 0.0f)) ? 1.0f : nvfp4 ? __fdiv_rn(2688.0f, a) : __fdiv_rn(a, 448.0f);
}

cudaError_t launch_scale_from_amax(const float *amax, float *out, int nvfp4, int zero_to_one,
                                   cudaStream_t stream)
{
    return launch_pdl(scale_from_amax_kernel, 1, 1, 0, stream, amax, out, nvfp4, zero_to_one);
}

}  // namespace rq
