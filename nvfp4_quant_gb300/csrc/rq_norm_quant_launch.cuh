// rq_norm_quant_launch.cuh -- configuration choice and persistent-grid launch
// of add_rmsnorm_quant_kernel.  Included by one translation unit per dtype.
#pragma once

#include <atomic>

#include "rq_norm_quant.cuh"

namespace rq {

constexpr int kMaxDevices = 64;

// Resident CTAs per SM of one kernel instantiation, cached per device.
template <typename Kern>
static int resident_ctas(Kern kern, int block, int dev, std::atomic<int> *cache)
{
    int v = dev < kMaxDevices ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (v > 0) return v;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, block, 0) != cudaSuccess || n < 1)
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
    const int per_sm = resident_ctas(kern, S::kBlock, dev, occ_cache);
    const int64_t groups = (p.rows + S::kRowsPerCta - 1) / S::kRowsPerCta;
    const int64_t full = (int64_t)device_sms(dev) * per_sm;
    const int grid = (int)(groups < full ? groups : full);
    kern<<<grid, S::kBlock, 0, stream>>>(p);
    return cudaGetLastError();
}

// Thread-group shape by row length (nvec 16-byte vectors per row): the
// smallest listed G x VPT that covers the row.
template <typename DT, int MODE>
cudaError_t launch_add_rmsnorm(const NormQuantParams &p, cudaStream_t stream)
{
    const int n = p.nvec;
    if (n <= 16) return launch_cfg<DT, 8, 2, MODE>(p, stream);
    if (n <= 64) return launch_cfg<DT, 32, 2, MODE>(p, stream);
    if (n <= 128) return launch_cfg<DT, 32, 4, MODE>(p, stream);
    if (n <= 256) return launch_cfg<DT, 64, 4, MODE>(p, stream);
    if (n <= 512) return launch_cfg<DT, 128, 4, MODE>(p, stream);
    if (n <= 896) return launch_cfg<DT, 128, 7, MODE>(p, stream);
    if (n <= 1024) return launch_cfg<DT, 128, 8, MODE>(p, stream);
    if (n <= 2048) return launch_cfg<DT, 256, 8, MODE>(p, stream);
    return launch_cfg<DT, 512, 8, MODE>(p, stream);  // n <= 4096 (hidden <= 32768)
}

}  // namespace rq

#define RQ_INSTANTIATE_NORM_QUANT(DT)                                                          \
    template cudaError_t rq::launch_add_rmsnorm<DT, rq::MODE_FP8>(const rq::NormQuantParams &, \
                                                                  cudaStream_t);               \
    template cudaError_t rq::launch_add_rmsnorm<DT, rq::MODE_NVFP4>(                           \
        const rq::NormQuantParams &, cudaStream_t);                                            \
    template cudaError_t rq::launch_add_rmsnorm<DT, rq::MODE_AMAX>(const rq::NormQuantParams &, \
                                                                   cudaStream_t);              \
    template cudaError_t rq::launch_add_rmsnorm<DT, rq::MODE_FP8_ROW>(                         \
        const rq::NormQuantParams &, cudaStream_t);
