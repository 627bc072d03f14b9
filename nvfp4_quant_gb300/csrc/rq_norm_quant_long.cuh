// rq_norm_quant_long.cuh -- the fused residual add + RMSNorm + quant kernel
// for long rows: above 32768 elements (no register shape reaches them), and
// above 16384 with more rows than SMs (where it measured faster than the
// shared-memory staged kernel and the 512 x 8 register shape).
//
// Such a row fits neither a thread group's registers nor, past 16384
// elements, a CTA's shared memory at useful occupancy, so a CTA of kLongThreads threads owns one row at
// a time and makes two passes over global memory.  Pass 1 loads x and the
// residual, forms residual' = dt(x + r), stores it and sums its squares.  After
// the row reduction, pass 2 reads back the residual' vectors the thread itself
// stored (the row was just written, so the reads are served by L2; no other
// thread's data is needed, so there is no barrier), normalises and quantises
// exactly as the other kernels do (same pairing of NVFP4 block halves in
// neighbouring lanes, same stores).  Where nothing is written back (the amax
// and gated modes) pass 2 forms residual' (or the gated value
// g = dt(x * dt(silu(z)))) again from the inputs, with the same operations.
// The per-token mode adds a third pass for the codes after the row maximum.
#pragma once

#include "rq_norm_quant.cuh"

namespace rq {

constexpr int kLongThreads = 512;
constexpr int kLongUnroll = 2;  // vectors per thread whose loads are issued together

template <typename DT, int MODE, bool kFast>
__device__ __forceinline__ void long_body(const NormQuantParams &p, float (*red)[kLongThreads / 32],
                                          const uint16_t *gtab)
{
    constexpr int T = kLongThreads;
    constexpr int kWarps = T / 32;
    // residual' is stored in pass 1 and read back in pass 2
    constexpr bool kWrites = MODE != MODE_AMAX && !is_gated<MODE>();
    const int tid = threadIdx.x;
    const int nvec = p.nvec;
    const int iters = (nvec + T - 1) / T;  // the same for every thread: shuffles stay converged
    const int64_t H = p.hidden;
    const uint8_t *w = static_cast<const uint8_t *>(p.w);

    const float scale = (MODE == MODE_FP8 || is_nvfp4<MODE>()) ? ld_f32(p.scale) : 1.0f;
    const Divisor by_scale(scale);
    const Divisor by_six(6.0f);
    const bool sf_words = (p.hidden % 64) == 0;
    float amax_acc = 0.0f;
    int parity = 0;

    constexpr int U = kLongUnroll;
    const uint8_t *px = static_cast<const uint8_t *>(p.x);
    const uint8_t *pr = static_cast<const uint8_t *>(p.res_in);
    auto at = [&](int64_t row, int k) { return (row * H + (int64_t)k * 8) * 2; };
    // residual' (or g) from the loaded x and residual (gate) vectors
    auto form = [&](uint4 xv, uint4 rv) {
        if (is_gated<MODE>())  // bf16: the gate table (filled by the kernel)
            return mul8<DT>(xv, std::is_same<DT, BF16>::value ? gate8_bf16(rv, gtab) : silu_gate8<DT>(rv));
        float a[8], b[8];
        unpack8<DT>(xv, a);
        unpack8<DT>(rv, b);
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] = __fadd_rn(a[e], b[e]);
        return pack8<DT>(a);
    };
    // pass 2 and 3: the values pass 1 formed for vectors i0 .. i0 + U - 1 of
    // this thread, read back or formed again (the loads of all U first)
    auto again = [&](int64_t row, int i0, uint4 (&sv)[U]) {
        uint4 xv[U], rv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int k = (i0 + u) * T + tid;
            const bool ok = i0 + u < iters && k < nvec;
            if (kWrites) {
                sv[u] = ok ? ld_stream16(static_cast<const uint8_t *>(p.res_out) + at(row, k))
                           : make_uint4(0, 0, 0, 0);
            } else {
                xv[u] = ok ? ld_stream16(px + at(row, k)) : make_uint4(0, 0, 0, 0);
                rv[u] = ok ? ld_stream16(pr + at(row, k)) : make_uint4(0, 0, 0, 0);
            }
        }
        if (!kWrites) {
#pragma unroll
            for (int u = 0; u < U; ++u) sv[u] = form(xv[u], rv[u]);
        }
    };
    // y = dt((s * rstd) * w) of vector k
    auto norm = [&](uint4 sv, int k, float rstd, float (&y)[8]) {
        float s[8], wf[8];
        unpack8<DT>(sv, s);
        unpack8<DT>(ld_keep16(w + (int64_t)k * 16), wf);
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(__fmul_rn(s[e], rstd), wf[e]);
        return pack8<DT>(y);
    };

    for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
        // ---- pass 1: residual' (stored), its squares; the loads of U
        // vectors first (the stores go to other addresses than these loads)
        float ss = 0.0f;
        for (int i0 = 0; i0 < iters; i0 += U) {
            uint4 xv[U], rv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = (i0 + u) * T + tid;
                const bool ok = i0 + u < iters && k < nvec;
                xv[u] = ok ? ld_stream16(px + at(row, k)) : make_uint4(0, 0, 0, 0);
                rv[u] = ok ? ld_stream16(pr + at(row, k)) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int k = (i0 + u) * T + tid;
                if (i0 + u < iters && k < nvec) {
                    const uint4 sv = form(xv[u], rv[u]);
                    if (kWrites) st16(static_cast<uint8_t *>(p.res_out) + at(row, k), sv);
                    float a[8];
                    unpack8<DT>(sv, a);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss = __fmaf_rn(a[e], a[e], ss);  // squares are exact
                }
            }
        }
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
        for (int i0 = 0; i0 < iters; i0 += U) {
            uint4 sv[U];
            again(row, i0, sv);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (i0 + u >= iters) break;  // the same for every thread
                const int k = (i0 + u) * T + tid;
                const bool ok = k < nvec;
                float y[8];
                uint4 yv = make_uint4(0, 0, 0, 0);
                if (ok) yv = norm(sv[u], k, rstd, y);
                if (MODE != MODE_AMAX && p.norm_out != nullptr && ok)
                    st16(static_cast<uint8_t *>(p.norm_out) + at(row, k), yv);
                unpack8<DT>(yv, y);  // quantise from the dtype-rounded norm output
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
                } else if (ok) {  // per-token FP8 (its row maximum first) or amax
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        if (MODE == MODE_FP8_ROW) row_amax = fmaxf(row_amax, fabsf(y[e]));
                        else amax_acc = fmaxf(amax_acc, fabsf(y[e]));
                    }
                }
            }
        }

        if (MODE == MODE_FP8_ROW) {
            // ---- pass 3: the codes at scale = row maximum / 448 (1 for a
            // zero row), from y formed again as in pass 2
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
            for (int i0 = 0; i0 < iters; i0 += U) {
                uint4 sv[U];
                again(row, i0, sv);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int k = (i0 + u) * T + tid;
                    if (i0 + u < iters && k < nvec) {
                        float y[8], v[8];
                        unpack8<DT>(norm(sv[u], k, rstd, y), y);
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
    }

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
__global__ void __launch_bounds__(kLongThreads)
add_rmsnorm_quant_long_kernel(const NormQuantParams p)
{
    __shared__ float red[2][kLongThreads / 32];
    // gated bf16: the gate table, filled before the wait (no global access)
    constexpr bool kGateTab = is_gated<MODE>() && std::is_same<DT, BF16>::value;
    __shared__ __align__(16) uint16_t gtab[kGateTab ? 2 * kGateHalf : 8];
    pdl_trigger();
    if (kGateTab) {
        gate_table_fill(gtab);
        __syncthreads();
    }
    pdl_wait();
    if (MODE == MODE_FP8 && !Divisor(ld_f32(p.scale)).fast)
        long_body<DT, MODE, false>(p, red, gtab);
    else
        long_body<DT, MODE, true>(p, red, gtab);
}

}  // namespace rq
