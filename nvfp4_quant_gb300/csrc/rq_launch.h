// rq_launch.h -- host-side launch interface between the C ABI (rq_api.cu) and
// the kernel translation units.  Internal to librq.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rq {

struct BF16;
struct FP16;

struct NormQuantParams {
    const void *x;
    const void *res_in;
    void *res_out;
    const void *w;
    void *norm_out;      // may be null
    uint8_t *q;          // FP8 codes [rows, H] or NVFP4 packed [rows, H/2]
    uint8_t *sf;         // NVFP4 block scales (layout below)
    const float *scale;  // FP8 dequant scale or NVFP4 global scale
    float *amax;         // amax-mode output
    float *row_scales;   // per-row FP8 scales [rows] (per-token mode)
    float eps;
    int64_t rows;
    int hidden;
    int nvec;            // hidden / 8
    int sf_col_tiles;    // swizzled scales: tiles of 4 block columns per row of tiles,
                         // ceil(H / 64)
};

struct QKParams {
    const void *q;
    const void *k;
    int64_t q_stride;    // elements between tokens
    int64_t k_stride;
    int64_t n_tokens;
    int hq, hk;
    const void *qw;
    const void *kw;
    float eps;
    const int32_t *pos;
    const float *cos_sin;
    int64_t max_pos;
    const float *q_scale;
    const float *k_scale;
    uint8_t *q_out;
    uint8_t *k_out;
    const int64_t *k_slots;  // null: K dense [T, Hk, D]; else K goes to pool row k_slots[t]
    int64_t num_slots;       // rows of the K pool
    int rope_dim;            // rotated elements at the end of each head (QK_MIXED; else D)
    float *q_amax;           // QK_AMAX outputs (may be the same address)
    float *k_amax;
    float nz;                // -0.0f, passed at run time (see mul2_unfused)
};

// What the Q/K kernel writes.  QK_STORE: FP8 codes of Q and K (K dense or to
// pool rows by slot).  QK_AMAX: nothing but max |o| over Q and over K.
// QK_MIXED: the RoPE on the last rope_dim elements of each head only; Q's FP8
// codes dense, K to pool rows by slot as [E4M3 of the first D - rope_dim
// elements | the last rope_dim elements as dtype values].
enum QKMode { QK_STORE = 0, QK_AMAX = 1, QK_MIXED = 2 };

// MODE_NVFP4 writes the block scales row-major [rows, H/16]; MODE_NVFP4_SWZ
// writes them in the 128 x 4-tile layout of block-scaled GEMMs (sf_offset).
// MODE_GATED_NVFP4 replaces the residual add by the gate
// g = dt(x * dt(silu(z))) (z in res_in; nothing written back) and quantises
// like MODE_NVFP4; MODE_GATED_NVFP4_SWZ likewise, with swizzled scales.
enum QuantMode {
    MODE_FP8 = 0,
    MODE_NVFP4 = 1,
    MODE_AMAX = 2,
    MODE_FP8_ROW = 3,
    MODE_NVFP4_SWZ = 4,
    MODE_GATED_NVFP4 = 5,
    MODE_GATED_NVFP4_SWZ = 6
};

template <int MODE>
__host__ __device__ constexpr bool is_nvfp4()
{
    return MODE == MODE_NVFP4 || MODE == MODE_NVFP4_SWZ || MODE == MODE_GATED_NVFP4 ||
           MODE == MODE_GATED_NVFP4_SWZ;
}

template <int MODE>
__host__ __device__ constexpr bool is_gated()
{
    return MODE == MODE_GATED_NVFP4 || MODE == MODE_GATED_NVFP4_SWZ;
}

template <int MODE>
__host__ __device__ constexpr bool is_swizzled()
{
    return MODE == MODE_NVFP4_SWZ || MODE == MODE_GATED_NVFP4_SWZ;
}

// SM count of device `dev` (cached).
int device_sms(int dev);

// Launch with programmatic stream serialisation allowed: the kernel's CTAs may
// be scheduled before the previous kernel in the stream has finished (each
// kernel waits for it with pdl_wait() before touching global memory).  Under
// stream capture this records a programmatic edge in the graph.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                       cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <typename DT, int MODE>
cudaError_t launch_add_rmsnorm(const NormQuantParams &p, cudaStream_t stream);

template <typename DT, int QMODE>
cudaError_t launch_qk_rmsnorm_rope(const QKParams &p, cudaStream_t stream);

// out = amax / 448 (nvfp4 == 0) or 2688 / amax (nvfp4 == 1); with
// zero_to_one, a zero amax gives 1.  out may equal amax.
cudaError_t launch_scale_from_amax(const float *amax, float *out, int nvfp4, int zero_to_one,
                                   cudaStream_t stream);

}  // namespace rq
