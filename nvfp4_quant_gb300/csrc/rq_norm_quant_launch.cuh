// rq_norm_quant_launch.cuh -- configuration choice and persistent-grid launch
// of add_rmsnorm_quant_kernel.  Included by one translation unit per dtype.
#pragma once

#include <atomic>

#include "rq_norm_quant.cuh"
#include "rq_norm_quant_long.cuh"
#include "rq_norm_quant_staged.cuh"
#include "rq.h"

namespace rq {

constexpr int kMaxDevices = 64;

// Resident CTAs per SM of one kernel instantiation, cached per device.
// A kernel with more than 48 KB of dynamic shared memory is first allowed it;
// 0 if that is refused.
template <typename Kern>
static int resident_ctas(Kern kern, int block, int dev, std::atomic<int> *cache, int smem = 0)
{
    int v = dev < kMaxDevices ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (v > 0) return v;
    int n = 0;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, block, smem) != cudaSuccess || n < 1)
        n = 1;
    if (dev < kMaxDevices) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

template <typename DT, int G, int VPT, int MODE>
static cudaError_t launch_cfg(const NormQuantParams &p, cudaStream_t stream)
{
    using S = GroupShape<G>;
    static std::atomic<int> occ_cache[kMaxDevices];
    auto kern = add_rmsnorm_quant_kernel<DT, G, VPT, MODE>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    constexpr int smem = dynamic_smem_bytes<DT, G, MODE>();
    const int per_sm = resident_ctas(kern, S::kBlock, dev, occ_cache, smem);
    if (per_sm < 1) return cudaErrorInvalidConfiguration;  // the shared memory was refused
    const int64_t groups = (p.rows + S::kRowsPerCta - 1) / S::kRowsPerCta;
    const int64_t full = (int64_t)device_sms(dev) * per_sm;
    const int grid = (int)(groups < full ? groups : full);
    return launch_pdl(kern, grid, S::kBlock, smem, stream, p);
}

// Long rows through shared memory: 4 * hidden bytes of dynamic shared memory
// per CTA; the resident-CTA count is cached per device for the last row
// length, the pair (shared memory bytes, CTAs per SM) in one 64-bit atomic so
// that concurrent callers never pair one length's count with another's.
template <typename DT, int MODE>
static cudaError_t launch_staged(const NormQuantParams &p, cudaStream_t stream)
{
    static std::atomic<uint64_t> occ[kMaxDevices];
    static std::atomic<int> attr_set[kMaxDevices];
    auto kern = add_rmsnorm_quant_staged_kernel<DT, MODE>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int smem = 32 * p.nvec;
    const int d = dev < kMaxDevices ? dev : 0;
    if (!attr_set[d].load(std::memory_order_relaxed)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 32 * kStagedMaxNvec);
        if (e != cudaSuccess) return e;
        attr_set[d].store(1, std::memory_order_relaxed);
    }
    const uint64_t cached = occ[d].load(std::memory_order_relaxed);
    int per_sm = (uint32_t)(cached >> 32) == (uint32_t)smem ? (int)(uint32_t)cached : 0;
    if (per_sm <= 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kStagedThreads, smem) !=
                cudaSuccess || per_sm < 1)
            per_sm = 1;
        occ[d].store(((uint64_t)(uint32_t)smem << 32) | (uint32_t)per_sm, std::memory_order_relaxed);
    }
    const int64_t full = (int64_t)device_sms(dev) * per_sm;
    const int grid = (int)(p.rows < full ? p.rows : full);
    return launch_pdl(kern, grid, kStagedThreads, smem, stream, p);
}

// The two-pass kernel (rows above 16384 elements with more rows than SMs, and
// every row above 32768): one CTA of kLongThreads per row, persistent grid.
template <typename DT, int MODE>
static cudaError_t launch_long(const NormQuantParams &p, cudaStream_t stream)
{
    static std::atomic<int> occ_cache[kMaxDevices];
    auto kern = add_rmsnorm_quant_long_kernel<DT, MODE>;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int per_sm = resident_ctas(kern, kLongThreads, dev, occ_cache);
    const int64_t full = (int64_t)device_sms(dev) * per_sm;
    const int grid = (int)(p.rows < full ? p.rows : full);
    return launch_pdl(kern, grid, kLongThreads, 0, stream, p);
}

// Thread-group shape by row length (nvec 16-byte vectors per row): with at
// most one row per SM, a wide group (256 or 512 threads per row); otherwise
// the smallest listed G x VPT that covers the row.  Rows of 8200 to 16384
// elements go through shared memory when there are at least two rows per SM
// (16384-element rows: 0.82 of the copy bandwidth staged against 0.75
// register-resident).  Longer rows with more rows than SMs, and all rows above
// 32768, take the two-pass kernel (rq_norm_quant_long.cuh), which beat both
// on GB300: 1024 x 20480 NVFP4 with norm out 38.3 us against 46.7 staged,
// 1000 x 24576 43.0 against 54.8, 2048 x 32768 100.8 against 106.0 for 512 x 8.
// With at most one row per SM the wide register shapes stay faster.
template <typename DT, int MODE>
cudaError_t launch_add_rmsnorm(const NormQuantParams &p, cudaStream_t stream)
{
    const int n = p.nvec;
    int dev = 0;
    if (n > 4096) return launch_long<DT, MODE>(p, stream);  // hidden above 32768
    // At most one row per SM: one CTA per row either way, so give each row
    // more threads and each thread fewer vectors (a shorter serial chain per
    // thread; measured on GB300 in a CUDA graph, the [64, 8192] fp16 NVFP4
    // tail with norm out went from 3.96 to 2.95 us).
    if (n > 256 && cudaGetDevice(&dev) == cudaSuccess && p.rows <= (int64_t)device_sms(dev)) {
        if (n <= 512) return launch_cfg<DT, 256, 2, MODE>(p, stream);
        if (n <= 1024) return launch_cfg<DT, 512, 2, MODE>(p, stream);
        if (n <= 2048) return launch_cfg<DT, 512, 4, MODE>(p, stream);
        return launch_cfg<DT, 512, 8, MODE>(p, stream);
    }
    // The gate's table lookups and SiLU make the gated call's chain per
    // vector long: more, shorter threads per row hide it better (16,384 x 7168
    // bf16: 448 x 2 at 28 warps per SM 155 us, 128 x 7 at 12 warps 168 us,
    // 512 x 2 at 64 warps 174 us).  This shape also takes fp16 gates from a
    // table (80 KB of shared memory per CTA).
    if constexpr (is_gated<MODE>()) {
        if (n > 512 && n <= 896) return launch_cfg<DT, 448, 2, MODE>(p, stream);
    }
    if (n <= 16) return launch_cfg<DT, 8, 2, MODE>(p, stream);
    if (n <= 64) return launch_cfg<DT, 32, 2, MODE>(p, stream);
    if (n <= 128) return launch_cfg<DT, 32, 4, MODE>(p, stream);
    if (n <= 256) return launch_cfg<DT, 64, 4, MODE>(p, stream);
    if (n <= 512) return launch_cfg<DT, 128, 4, MODE>(p, stream);
    if (n > 1024 && n <= 2048) {
        if (cudaGetDevice(&dev) == cudaSuccess && p.rows >= 2 * (int64_t)device_sms(dev))
            return launch_staged<DT, MODE>(p, stream);
    }
    if (n <= 896) return launch_cfg<DT, 128, 7, MODE>(p, stream);
    if (n <= 1024) return launch_cfg<DT, 128, 8, MODE>(p, stream);
    if (n <= 2048) return launch_cfg<DT, 256, 8, MODE>(p, stream);
    return launch_long<DT, MODE>(p, stream);  // above 16384 elements
}

}  // namespace rq

// One mode of one dtype (the build compiles each mode in its own translation
// unit, in parallel, with -DRQ_MODE=<mode>), or all of them.
#define RQ_INSTANTIATE_MODE(DT, MODE)                                                          \
    template cudaError_t rq::launch_add_rmsnorm<DT, MODE>(const rq::NormQuantParams &, cudaStream_t);

#define RQ_INSTANTIATE_NORM_QUANT(DT)                                                          \
    template cudaError_t rq::launch_add_rmsnorm<DT, rq::MODE_FP8>(const rq::NormQuantParams &, \
                                                                  cudaStream_t);               \
    template cudaError_t rq::launch_add_rmsnorm<DT, rq::MODE_NVFP4>(                           \
        const rq::NormQuantParams &, cudaStream_t);                                            \
    template cudaError_t rq::launch_add_rmsnorm<DT, rq::MODE_AMAX>(const rq::NormQuantParams &, \
                                                                   cudaStream_t);              \
    template cudaError_t rq::launch_add_rmsnorm<DT, rq::MODE_FP8_ROW>(                         \
        const rq::NormQuantParams &, cudaStream_t);                                            \
    template cudaError_t rq::launch_add_rmsnorm<DT, rq::MODE_NVFP4_SWZ>(                       \
        const rq::NormQuantParams &, cudaStream_t);                                            \
    template cudaError_t rq::launch_add_rmsnorm<DT, rq::MODE_GATED_NVFP4>(                     \
        const rq::NormQuantParams &, cudaStream_t);                                            \
    template cudaError_t rq::launch_add_rmsnorm<DT, rq::MODE_GATED_NVFP4_SWZ>(                 \
        const rq::NormQuantParams &, cudaStream_t);
