// rq_norm_quant.cuh -- the fused residual add + RMSNorm (+ norm output) +
// FP8 / NVFP4 kernel, and its amax-calibration variant.
//
// Prior art: "[Performance]: Fuse local NVFP4 tail after NCCL fallback"
// (TensorRT-LLM issue 17900), Proposal: one launch for residual + RMSNorm +
// NVFP4 instead of separate kernels; "Add NanoJet backend for AutoDeploy
// prefill-only FP8 inference", Description: RMSNorm with FP8 quantisation in
// the epilogue.  The design below is ours, for GB300.
//
// Work mapping.  A row of `hidden` elements is split into nvec = hidden / 8
// vectors of 16 bytes.  A row group of G threads owns one row; thread t of the
// group holds vectors t, t + G, ..., t + (VPT-1) G, so each warp-wide access
// touches consecutive 16-byte vectors (fully coalesced) and the two vectors
// of one 16-element NVFP4 block sit in neighbouring lanes.  G <= 32 packs
// 32 / G rows into a warp; G > 32 spans warps of one CTA.  The grid is
// persistent: each CTA walks row groups with a grid stride, keeping the
// weight in registers for all its rows.
//
// Per row: 16-byte loads of x and residual -> fp32 add -> round to the dtype
// -> store residual' -> fp32 sum of squares of the rounded values (shuffle
// tree, then shared memory across warps) -> rstd with IEEE div / sqrt ->
// y = dt((s * rstd) * w) -> optional norm_out store -> quantise from the
// rounded y.
#pragma once

#include "rq_device.cuh"
#include "rq_launch.h"

#include <type_traits>

namespace rq {

template <int G>
struct GroupShape {
    static constexpr int kBlock = G >= 128 ? G : 128;    // threads per CTA
    static constexpr int kRowsPerCta = kBlock / G;
    static constexpr int kWarps = kBlock / 32;
    static constexpr int kWarpsPerGroup = G > 32 ? G / 32 : 1;
    // per-warp partial sums in shared memory: a row of them per parity,
    // padded to whole 16-byte vectors (the padding holds zeros)
    static constexpr int kRedStride = (kWarps + 3) & ~3;
};

// Byte offset of the block scale of (row, block column c).  Linear layout:
// row-major [rows, H/16].  Swizzled layout (the one a block-scaled NVFP4 GEMM
// reads): the scale matrix, padded to 128-row and 4-column multiples, is cut
// into 128 x 4 tiles of 512 bytes, the row of tiles outermost; inside a tile
// (r, c) sits at 16 * (r % 32) + 4 * (r / 32) + c.  In both, the four scales
// of block columns 4j..4j+3 of a row are four consecutive bytes.
template <bool kSwz>
__device__ __forceinline__ int64_t sf_offset(const NormQuantParams &p, int64_t row, int c)
{
    if (!kSwz) return row * (p.hidden / 16) + c;
    return ((row >> 7) * p.sf_col_tiles + (c >> 2)) * 512 + (row & 31) * 16 + ((row >> 5) & 3) * 4 +
           (c & 3);
}

// Swizzled layout: zero bytes for the rows that pad the last row of tiles,
// one 32-bit word per (row, column tile), spread over the whole grid.  (The
// padding columns of real rows are written by the thread that stores the
// row's last block scale.)
__device__ __forceinline__ void sf_zero_pad_rows(const NormQuantParams &p)
{
    const int64_t first = p.rows;
    const int64_t words = ((first + 127) / 128 * 128 - first) * p.sf_col_tiles;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < words;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = first + i / p.sf_col_tiles;
        const int ct = (int)(i % p.sf_col_tiles);
        st4(p.sf + sf_offset<true>(p, r, ct * 4), 0u);
    }
}

// Swizzled layout: where the row's bytes of its first tile start (the row's
// part of sf_offset); block column c adds (c / 4) * 512 + c % 4.  (Computing
// it once per row at the top of the row loop, instead of at each store, made
// the 16,384 x 7168 call 11 % slower: the loads of the row issue later.)
__device__ __forceinline__ uint8_t *sf_swizzled_row(const NormQuantParams &p, int64_t row)
{
    return p.sf + (((row >> 7) * p.sf_col_tiles) << 9) + ((row & 31) << 4) + (((row >> 5) & 3) << 2);
}

// Stores the block scale sfc of block column c = k / 2 (k = this lane's
// vector index; the lanes of vectors k and k + 1 hold the same scale).  With
// whole groups of four columns (hidden % 64 == 0) the lane of k % 8 == 0
// stores the four scales of its group as one word, gathered from the lanes
// 2, 4 and 6 above it; otherwise each even-k lane stores its byte, and in the
// swizzled layout the lane of the last column also zeroes the padding
// columns after it.  Every lane of the warp must call this (shuffles).
template <bool kSwz>
__device__ __forceinline__ void store_block_scale(const NormQuantParams &p, int64_t row, int k,
                                                  bool ok, uint32_t sfc, bool sf_words)
{
    // linear: the row's scales start at row * H/16
    uint8_t *base = kSwz ? sf_swizzled_row(p, row) : p.sf + row * (int64_t)(p.hidden / 16);
    auto at = [&](int c) { return kSwz ? base + ((c >> 2) << 9) + (c & 3) : base + c; };
    if (sf_words) {
        const uint32_t b1 = __shfl_down_sync(0xFFFFFFFFu, sfc, 2);
        const uint32_t b2 = __shfl_down_sync(0xFFFFFFFFu, sfc, 4);
        const uint32_t b3 = __shfl_down_sync(0xFFFFFFFFu, sfc, 6);
        // a word starts at a column multiple of 4: k % 8 == 0, c = k / 2
        uint8_t *dst = kSwz ? base + ((k >> 3) << 9) : base + k / 2;
        if (ok && (k & 7) == 0) st4(dst, sfc | (b1 << 8) | (b2 << 16) | (b3 << 24));
    } else if (ok && (k & 1) == 0) {
        st1(at(k / 2), sfc);
        const int nb = p.hidden / 16;
        if (kSwz && k / 2 == nb - 1)
            for (int cc = nb; cc < p.sf_col_tiles * 4; ++cc) st1(at(cc), 0u);
    }
}

// Whether a shape takes fp16 gates from a table in dynamic shared memory (the
// gated call's 448 x 2 shape: two CTAs per SM either way), and its bytes.
template <typename DT, int G, int MODE>
__host__ __device__ constexpr bool gate_table_fp16()
{
    return is_gated<MODE>() && std::is_same<DT, FP16>::value && G == 448;
}

template <typename DT, int G, int MODE>
__host__ __device__ constexpr int dynamic_smem_bytes()
{
    return gate_table_fp16<DT, G, MODE>() ? 2 * kGateHalfF16 * 2 : 0;
}

// kFast: the FP8 divisor is in the range of the branch-free division (the
// kernel picks the body once; see Divisor).
template <typename DT, int G, int VPT, int MODE, bool kFast>
__device__ __forceinline__ void add_rmsnorm_quant_body(const NormQuantParams &p,
                                                       float (*red)[GroupShape<G>::kRedStride])
{
    using S = GroupShape<G>;
    const int tid = threadIdx.x;
    const int t = tid % G;
    const int grp = tid / G;
    const int nvec = p.nvec;
    const int64_t H = p.hidden;

    // gated bf16: the gate table in shared memory, computed (no global memory
    // access) while the previous kernel in the stream may still be running
    constexpr bool kGateTab = is_gated<MODE>() && std::is_same<DT, BF16>::value;
    __shared__ __align__(16) uint16_t gtab[kGateTab ? 2 * kGateHalf : 8];
    if (kGateTab) {
        gate_table_fill(gtab);
        __syncthreads();
    }
    // gated fp16 in the 448 x 2 shape: its table in dynamic shared memory
    constexpr bool kGateTab16 = gate_table_fp16<DT, G, MODE>();
    extern __shared__ __align__(16) uint16_t gtab16[];
    if (kGateTab16) {
        gate_table_fill_fp16(gtab16);
        __syncthreads();
    }
    pdl_wait();

    // weight vectors of this thread, kept for every row it processes
    uint4 wv[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int k = j * G + t;
        wv[j] = k < nvec ? ld_keep16(static_cast<const uint8_t *>(p.w) + (int64_t)k * 16)
                         : make_uint4(0, 0, 0, 0);
    }
    const float scale = (MODE == MODE_FP8 || is_nvfp4<MODE>()) ? ld_f32(p.scale) : 1.0f;
    const Divisor by_scale(scale);  // FP8: y / scale
    const Divisor by_six(6.0f);     // NVFP4: (gs * amax) / 6
    const bool sf_words = (p.hidden % 64) == 0;  // 4 block scales per 32-bit store
    // NVFP4: enc = scale / sf for each of the 256 E4M3 scale bytes (0 where
    // sf is 0), one correctly rounded division each, looked up per block
    __shared__ float enc_tab[is_nvfp4<MODE>() ? 256 : 1];
    if (is_nvfp4<MODE>()) {
        for (int c = tid; c < 256; c += S::kBlock) {
            const float sfv = e4m3_value(c);
            enc_tab[c] = sfv == 0.0f ? 0.0f : __fdiv_rn(scale, sfv);
        }
        __syncthreads();
    }
    float amax_acc = 0.0f;
    int parity = 0;

    for (int64_t base = (int64_t)blockIdx.x * S::kRowsPerCta; base < p.rows;
         base += (int64_t)gridDim.x * S::kRowsPerCta) {
        const int64_t row = base + grp;
        const bool row_ok = row < p.rows;
        const uint8_t *xrow = static_cast<const uint8_t *>(p.x) + row * H * 2;
        const uint8_t *rrow = static_cast<const uint8_t *>(p.res_in) + row * H * 2;

        // ---- loads: all of this thread's vectors before any use
        uint4 xv[VPT], sv[VPT];
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = j * G + t;
            if (row_ok && k < nvec) {
                xv[j] = ld_stream16(xrow + (int64_t)k * 16);
                sv[j] = ld_stream16(rrow + (int64_t)k * 16);
            } else {
                xv[j] = make_uint4(0, 0, 0, 0);
                sv[j] = make_uint4(0, 0, 0, 0);
            }
        }

        // ---- residual' = dt(x + r), stored (gated: g = dt(x * dt(silu(z))),
        // not stored); sum of squares of the rounded values, as two partial
        // sums (even and odd elements) in one packed fp32 FMA per pair
        float2 sq = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            float a[8];
            if (is_gated<MODE>()) {
                const bool ok = row_ok && j * G + t < nvec;
                // the gate rounded to the dtype: from the table (bf16) or the
                // fast SiLU with its exact path (fp16)
                const uint4 gate = kGateTab     ? gate8_bf16(sv[j], gtab)
                                   : kGateTab16 ? gate8_fp16(sv[j], gtab16)
                                                : silu_gate8<DT>(sv[j], ok);
                sv[j] = mul8<DT>(xv[j], gate);
            } else {
                float b[8];
                unpack8<DT>(xv[j], a);
                unpack8<DT>(sv[j], b);
#pragma unroll
                for (int e = 0; e < 8; ++e) a[e] = __fadd_rn(a[e], b[e]);
                sv[j] = pack8<DT>(a);
            }
            unpack8<DT>(sv[j], a);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 ai = make_float2(a[2 * i], a[2 * i + 1]);
                sq = __ffma2_rn(ai, ai, sq);  // squares are exact
            }
            const int k = j * G + t;
            if (MODE != MODE_AMAX && !is_gated<MODE>() && row_ok && k < nvec)
                st16(static_cast<uint8_t *>(p.res_out) + (row * H + (int64_t)k * 8) * 2, sv[j]);
        }

        // ---- row reduction
        float ss = __fadd_rn(sq.x, sq.y);
        if (G <= 32) {
            ss = group_sum<(G <= 32 ? G : 32)>(ss);
        } else {
            ss = group_sum<32>(ss);
            if ((tid & 31) == 0) red[parity][tid >> 5] = ss;
            __syncthreads();
            const int w0 = grp * S::kWarpsPerGroup;
            if constexpr (S::kWarpsPerGroup >= 8) {
                // one row per CTA (w0 = 0): the partials as 16-byte vectors,
                // added pairwise with packed adds (the padding adds +0)
                const float4 *r4 = reinterpret_cast<const float4 *>(red[parity]);
                float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int i = 0; i < S::kRedStride / 4; ++i) {
                    const float4 v = r4[i];
                    acc = __fadd2_rn(acc, make_float2(v.x, v.y));
                    acc = __fadd2_rn(acc, make_float2(v.z, v.w));
                }
                ss = __fadd_rn(acc.x, acc.y);
            } else {
                ss = 0.0f;
#pragma unroll
                for (int i = 0; i < S::kWarpsPerGroup; ++i) ss = __fadd_rn(ss, red[parity][w0 + i]);
            }
            parity ^= 1;
        }
        const float ms = __fdiv_rn(ss, (float)p.hidden);
        const float rstd = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, p.eps)));

        // ---- normalise, store, quantise
        float row_amax = 0.0f;  // per-token mode: max |y| of this thread's part of the row
        const float2 r2 = make_float2(rstd, rstd);
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int k = j * G + t;
            const bool ok = row_ok && k < nvec;
            float s[8], w[8], y[8];
            unpack8<DT>(sv[j], s);
            unpack8<DT>(wv[j], w);
            // (s * rstd) * w, each product rounded: packed pairs, except in the
            // swizzled NVFP4 mode, where the scalar form measured faster on GB300
            // (166 against 176 us on 16,384 x 7168; as with the swizzled row
            // offset above, the packed form delays the next row's loads)
            if (MODE == MODE_NVFP4_SWZ) {
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = __fmul_rn(__fmul_rn(s[e], rstd), w[e]);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 yi = __fmul2_rn(__fmul2_rn(make_float2(s[2 * i], s[2 * i + 1]), r2),
                                                 make_float2(w[2 * i], w[2 * i + 1]));
                    y[2 * i] = yi.x;
                    y[2 * i + 1] = yi.y;
                }
            }
            const uint4 yv = pack8<DT>(y);
            if (MODE != MODE_AMAX && p.norm_out != nullptr && ok)
                st16(static_cast<uint8_t *>(p.norm_out) + (row * H + (int64_t)k * 8) * 2, yv);
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
                const float enc = enc_tab[sfc];
                const float2 enc2 = make_float2(enc, enc);
                float v[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 vi = __fmul2_rn(make_float2(y[2 * i], y[2 * i + 1]), enc2);
                    v[2 * i] = vi.x;
                    v[2 * i + 1] = vi.y;
                }
                const uint32_t codes = e2m1x8(v);
                if (ok) st4(p.q + row * (H / 2) + (int64_t)k * 4, codes);
                store_block_scale<is_swizzled<MODE>()>(p, row, k, ok, sfc, sf_words);
            } else if (MODE == MODE_FP8_ROW) {
                sv[j] = yv;  // residual' is stored; keep the rounded y for the second pass
                if (ok) {
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
            // the row's absolute maximum, its scale amax / 448 (1 for a zero
            // row), then the codes from the rounded y kept in registers
            if (G <= 32) {
                row_amax = group_max<(G <= 32 ? G : 32)>(row_amax);
            } else {
                row_amax = group_max<32>(row_amax);
                if ((tid & 31) == 0) red[parity][tid >> 5] = row_amax;
                __syncthreads();
                const int w0 = grp * S::kWarpsPerGroup;
                row_amax = 0.0f;
#pragma unroll
                for (int i = 0; i < S::kWarpsPerGroup; ++i) row_amax = fmaxf(row_amax, red[parity][w0 + i]);
                parity ^= 1;
            }
            const float rs = row_amax > 0.0f ? div_rn(row_amax, 448.0f) : 1.0f;
            const Divisor d(rs);
            if (row_ok && t == 0) p.row_scales[row] = rs;
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int k = j * G + t;
                float y[8], v[8];
                unpack8<DT>(sv[j], y);
                if (d.fast) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = div_by<true>(y[e], d);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = div_by<false>(y[e], d);
                }
                const uint2 c = e4m3x8(v);
                if (row_ok && k < nvec) st8(p.q + row * H + (int64_t)k * 8, c.x, c.y);
            }
        }
    }

    if (is_swizzled<MODE>()) sf_zero_pad_rows(p);

    if (MODE == MODE_AMAX) {
        // block maximum, then one atomic per CTA on the float's bit pattern
        // (non-negative floats order like their unsigned bits)
        float m = group_max<32>(amax_acc);
        __syncthreads();
        if ((tid & 31) == 0) red[0][tid >> 5] = m;
        __syncthreads();
        if (tid == 0) {
            float r = 0.0f;
            for (int i = 0; i < S::kWarps; ++i) r = fmaxf(r, red[0][i]);
            atomicMax(reinterpret_cast<unsigned int *>(p.amax), __float_as_uint(r));
        }
    }
}

// Register budget: the gated call's 448 x 2 shape is held to two CTAs per SM
// (70 registers).  The 128-thread shapes with 7 or 8 vectors per thread hold
// about 167 registers; past 170 only two CTAs fit per SM and the NVFP4 call on
// 16,384 x 7168 slows from 160 to 195 us, so they are held to three CTAs.
// Every other shape passes 0 (no minimum), which leaves ptxas its own
// occupancy heuristic: an explicit minimum of 1 lets it spend up to 255
// registers, and the 32 x 4 shape went from 96 to 152 registers (five CTAs per
// SM down to three) and 32,768 x 2048 from 95 to 107 us.
template <int G, int VPT>
constexpr int min_ctas_per_sm()
{
    return (G == 128 && VPT >= 7) ? 3 : (G == 448 && VPT == 2) ? 2 : 0;
}

template <typename DT, int G, int VPT, int MODE>
__global__ void __launch_bounds__(GroupShape<G>::kBlock, (min_ctas_per_sm<G, VPT>()))
add_rmsnorm_quant_kernel(const NormQuantParams p)
{
    using S = GroupShape<G>;
    __shared__ __align__(16) float red[2][S::kRedStride];
    if (S::kRedStride > S::kWarps && threadIdx.x < 2 * (S::kRedStride - S::kWarps)) {
        const int pad = S::kRedStride - S::kWarps;  // never written by a warp's partial
        red[threadIdx.x / pad][S::kWarps + threadIdx.x % pad] = 0.0f;
    }
    pdl_trigger();
    if (MODE == MODE_FP8) pdl_wait();  // before the scale load; the body waits in any case
    if (MODE == MODE_FP8 && !Divisor(ld_f32(p.scale)).fast)
        add_rmsnorm_quant_body<DT, G, VPT, MODE, false>(p, red);
    else
        add_rmsnorm_quant_body<DT, G, VPT, MODE, true>(p, red);
}

}  // namespace rq
