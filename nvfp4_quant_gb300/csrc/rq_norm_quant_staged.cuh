// rq_norm_quant_staged.cuh -- the fused residual add + RMSNorm + quant
// kernel for long rows (hidden 8200 to 16384, at least two rows per SM),
// staged through shared memory.
//
// Register-resident rows of this length need 64 KB and more of registers per
// row: one CTA per SM at most, or spills.  Here a CTA of kStagedThreads
// threads owns one row at a time and each thread copies its own 16-byte
// vectors of x and residual into shared memory with cp.async (waited with
// cp.async.wait_group, so no thread waits on another).  Pass 1 forms
// residual' = dt(x + r), stores it, writes it back over the residual slot and
// sums its squares; after the row reduction pass 2 normalises from shared
// memory and quantises exactly as the register-resident kernel does (same
// pairing of NVFP4 block halves in neighbouring lanes, same stores).  In the
// gated mode the residual slot holds the gate z and pass 1 forms
// g = dt(x * dt(silu(z))) there instead, without writing it back.
// Registers stay low, so shared memory (4 * hidden bytes per row) sets the
// number of rows in flight per SM: three at hidden 16384.
#pragma once

#include "rq_norm_quant.cuh"

namespace rq {

constexpr int kStagedThreads = 256;
// the longest row (in 16-byte vectors) the kernel's dynamic shared memory is
// allowed for: 32 bytes per vector (x and residual), 64 KB
constexpr int kStagedMaxNvec = 2048;

template <typename DT, int MODE, bool kFast>
__device__ __forceinline__ void staged_body(const NormQuantParams &p, uint4 *buf, float (*red)[kStagedThreads / 32])
{
    constexpr int T = kStagedThreads;
    constexpr int kWarps = T / 32;
    const int tid = threadIdx.x;
    const int nvec = p.nvec;
    const int iters = (nvec + T - 1) / T;  // the same for every thread: shuffles stay converged
    const int64_t H = p.hidden;
    uint4 *xs = buf;          // x, later the rounded y (per-token mode)
    uint4 *rs = buf + nvec;   // residual, then residual'
    const uint8_t *w = static_cast<const uint8_t *>(p.w);

    const float scale = (MODE == MODE_FP8 || is_nvfp4<MODE>()) ? ld_f32(p.scale) : 1.0f;
    const Divisor by_scale(scale);
    const Divisor by_six(6.0f);
    const bool sf_words = (p.hidden % 64) == 0;
    float amax_acc = 0.0f;
    int parity = 0;

    // the x slots are refilled with the next row as soon as pass 1 has read
    // them (not in per-token mode, which keeps the rounded y there)
    constexpr bool kEarlyX = MODE != MODE_FP8_ROW;
    auto stage = [&](int64_t r, uint4 *dst, const void *src_base) {
        if (r < p.rows) {
            const uint8_t *src = static_cast<const uint8_t *>(src_base) + r * H * 2;
            for (int i = 0; i < iters; ++i) {
                const int k = i * T + tid;
                if (k < nvec) cp_async16(dst + k, src + (int64_t)k * 16);
            }
        }
    };
    if (kEarlyX) stage(blockIdx.x, xs, p.x);

    for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
        if (!kEarlyX) stage(row, xs, p.x);
        stage(row, rs, p.res_in);
        cp_async_commit();
        cp_async_wait<0>();  // this thread's own vectors of the row

        // ---- pass 1: residual', its squares
        float ss = 0.0f;
        for (int i = 0; i < iters; ++i) {
            const int k = i * T + tid;
            if (k < nvec) {
                float a[8];
                uint4 sv;
                if (is_gated<MODE>()) {  // g = dt(x * dt(silu(z)))
                    sv = mul8<DT>(lds16(xs + k), silu_gate8<DT>(lds16(rs + k)));
                } else {
                    float b[8];
                    unpack8<DT>(lds16(xs + k), a);
                    unpack8<DT>(lds16(rs + k), b);
#pragma unroll
                    for (int e = 0; e < 8; ++e) a[e] = __fadd_rn(a[e], b[e]);
                    sv = pack8<DT>(a);
                }
                if (MODE != MODE_AMAX && !is_gated<MODE>())
                    st16(static_cast<uint8_t *>(p.res_out) + (row * H + (int64_t)k * 8) * 2, sv);
                sts16(rs + k, sv);
                unpack8<DT>(sv, a);
#pragma unroll
                for (int e = 0; e < 8; ++e) ss = __fmaf_rn(a[e], a[e], ss);  // squares are exact
            }
        }
        if (kEarlyX) stage(row + gridDim.x, xs, p.x);  // lands during the rest of this row
        ss = group_sum<32>(ss);
        if ((tid & 31) == 0) red[parity][tid >> 5] = ss;
        __syncthreads();
        ss = 0.0f;
#pragma unroll
        for (int i = 0; i < kWarps; ++i) ss = __fadd_rn(ss, red[parity][i]);
        parity ^= 1;
        const float ms = __fdiv_rn(ss, (float)p.hidden);
        const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, p.eps)));

        // ---- pass 2: normalise, store, quantise
        float row_amax = 0.0f;
        for (int i = 0; i < iters; ++i) {
            const int k = i * T + tid;
            const bool ok = k < nvec;
            float s[8], wf[8], y[8];
            unpack8<DT>(ok ? lds16(rs + k) : make_uint4(0, 0, 0, 0), s);
            unpack8<DT>(ok ? ld_keep16(w + (int64_t)k * 16) : make_uint4(0, 0, 0, 0), wf);
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(__fmul_rn(s[e], rstd), wf[e]);
            const uint4 yv = pack8<DT>(y);
            if (MODE != MODE_AMAX && p.norm_out != nullptr && ok)
                st16(static_cast<uint8_t *>(p.norm_out) + (row * H + (int64_t)k * 8) * 2, yv);
            unpack8<DT>(yv, y);
            if (MODE == MODE_FP8) {
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = div_by<kFast>(y[e], by_scale);
                const uint2 c = e4m3x8(v);
                if (ok) st8(p.q + row * H + (int64_t)k * 8, c.x, c.y);
            } else if (is_nvfp4<MODE>()) {
                float m = 0.0f;
#pragma unroll
                for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(y[e]));
                const float a = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));  // 16-element block
                const float t2 = div_by<true>(__fmul_rn(scale, a), by_six);
                const uint32_t sfc = e4m3x2(t2, 0.0f) & 0xFFu;
                const float sfv = e4m3_value(sfc);
                const float enc = sfv == 0.0f ? 0.0f : __fdiv_rn(scale, sfv);
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = __fmul_rn(y[e], enc);
                const uint32_t codes = e2m1x8(v);
                if (ok) st4(p.q + row * (H / 2) + (int64_t)k * 4, codes);
                store_block_scale<is_swizzled<MODE>()>(p, row, k, ok, sfc, sf_words);
            } else if (MODE == MODE_FP8_ROW) {
                if (ok) {
                    sts16(xs + k, yv);  // the rounded y, for the pass after the row maximum
#pragma unroll
                    for (int e = 0; e < 8; ++e) row_amax = fmaxf(row_amax, fabsf(y[e]));
                }
            } else {  // MODE_AMAX
                if (ok) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) amax_acc = fmaxf(amax_acc, fabsf(y[e]));
                }
            }
        }

        if (MODE == MODE_FP8_ROW) {
            row_amax = group_max<32>(row_amax);
            if ((tid & 31) == 0) red[parity][tid >> 5] = row_amax;
            __syncthreads();
            row_amax = 0.0f;
#pragma unroll
            for (int i = 0; i < kWarps; ++i) row_amax = fmaxf(row_amax, red[parity][i]);
            parity ^= 1;
            const float rsc = row_amax > 0.0f ? div_rn(row_amax, 448.0f) : 1.0f;
            const Divisor d(rsc);
            if (tid == 0) p.row_scales[row] = rsc;
            for (int i = 0; i < iters; ++i) {
                const int k = i * T + tid;
                if (k < nvec) {
                    float y[8], v[8];
                    unpack8<DT>(lds16(xs + k), y);
                    if (d.fast) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = div_by<true>(y[e], d);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = div_by<false>(y[e], d);
                    }
                    const uint2 c = e4m3x8(v);
                    st8(p.q + row * H + (int64_t)k * 8, c.x, c.y);
                }
            }
        }
    }

    cp_async_commit();
    cp_async_wait<0>();  // nothing may stay in flight at exit

    if (is_swizzled<MODE>()) sf_zero_pad_rows(p);

    if (MODE == MODE_AMAX) {
        float m = group_max<32>(amax_acc);
        __syncthreads();
        if ((tid & 31) == 0) red[0][tid >> 5] = m;
        __syncthreads();
        if (tid == 0) {
            float r = 0.0f;
            for (int i = 0; i < kWarps; ++i) r = fmaxf(r, red[0][i]);
            atomicMax(reinterpret_cast<unsigned int *>(p.amax), __float_as_uint(r));
        }
    }
}

template <typename DT, int MODE>
__global__ void __launch_bounds__(kStagedThreads)
add_rmsnorm_quant_staged_kernel(const NormQuantParams p)
{
    __shared__ float red[2][kStagedThreads / 32];
    extern __shared__ uint4 buf[];  // 2 * nvec vectors: x then residual
    pdl_trigger();
    pdl_wait();
    if (MODE == MODE_FP8 && !Divisor(ld_f32(p.scale)).fast)
        staged_body<DT, MODE, false>(p, buf, red);
    else
        staged_body<DT, MODE, true>(p, buf, red);
}

}  // namespace rq
