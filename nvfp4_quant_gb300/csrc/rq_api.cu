// rq_api.cu -- the C ABI of librq (declared in include/rq.h): argument checks,
// dispatch by dtype, launch, status codes.  Every check runs before the first
// CUDA call, so a rejected call touches neither the device nor the stream.
#include "rq.h"
#include "rq_launch.h"

#include <atomic>
#include <cstdio>
#include <cstring>

namespace {

thread_local char g_last_error[256] = "";

constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];

rq_status cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return RQ_OK;
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s", cudaGetErrorName(e),
                  cudaGetErrorString(e));
    return RQ_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

struct Span {
    uintptr_t lo, hi;  // [lo, hi); empty when lo == hi
};

Span span(const void *p, int64_t bytes)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Span{a, a + (uintptr_t)(p ? bytes : 0)};
}

bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

// true if any output overlaps another output or any input; `allow` names one
// (output, input) pair that may coincide exactly (the in-place residual).
bool bad_alias(const Span *outs, int n_out, const Span *ins, int n_in, int allow_out = -1,
               int allow_in = -1)
{
    for (int i = 0; i < n_out; ++i) {
        for (int j = i + 1; j < n_out; ++j)
            if (overlap(outs[i], outs[j])) return true;
        for (int j = 0; j < n_in; ++j) {
            if (!overlap(outs[i], ins[j])) continue;
            if (i == allow_out && j == allow_in && outs[i].lo == ins[j].lo && outs[i].hi == ins[j].hi)
                continue;
            return true;
        }
    }
    return false;
}

rq_status check_rows(int64_t rows, int64_t hidden, int dt)
{
    if (dt != RQ_BF16 && dt != RQ_FP16) return RQ_ERR_DTYPE;
    if (rows < 0 || hidden <= 0 || hidden % 16 != 0) return RQ_ERR_SHAPE;
    if (hidden > RQ_MAX_HIDDEN) return RQ_ERR_UNSUPPORTED;
    if (rows > (int64_t)1 << 40) return RQ_ERR_SHAPE;
    return RQ_OK;
}

rq::NormQuantParams make_params(const void *x, const void *res_in, void *res_out, const void *w,
                                float eps, const float *scale, uint8_t *q, uint8_t *sf,
                                void *norm_out, float *amax, int64_t rows, int64_t hidden)
{
    rq::NormQuantParams p;
    p.x = x;
    p.res_in = res_in;
    p.res_out = res_out;
    p.w = w;
    p.norm_out = norm_out;
    p.q = q;
    p.sf = sf;
    p.scale = scale;
    p.amax = amax;
    p.row_scales = nullptr;
    p.eps = eps;
    p.rows = rows;
    p.hidden = (int)hidden;
    p.nvec = (int)(hidden / 8);
    p.sf_col_tiles = (int)((hidden / 16 + 3) / 4);
    return p;
}

// Bytes of the NVFP4 block scales in either layout.
int64_t sf_bytes(int64_t rows, int64_t hidden, int swizzled)
{
    if (!swizzled) return rows * (hidden / 16);
    return (rows + 127) / 128 * 128 * ((hidden / 16 + 3) / 4 * 4);
}

template <int MODE>
rq_status launch_rows(const rq::NormQuantParams &p, rq_dtype dt, rq_stream_t stream)
{
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = dt == RQ_BF16 ? rq::launch_add_rmsnorm<rq::BF16, MODE>(p, s)
                                  : rq::launch_add_rmsnorm<rq::FP16, MODE>(p, s);
    return cuda_status(e);
}

}  // namespace

namespace rq {
int device_sms(int dev)
{
    int v = dev >= 0 && dev < kMaxDevices ? g_sms[dev].load(std::memory_order_relaxed) : 0;
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1) v = 1;
    if (dev >= 0 && dev < kMaxDevices) g_sms[dev].store(v, std::memory_order_relaxed);
    return v;
}
}  // namespace rq

namespace {

// Dynamic per-tensor scale: the amax pass accumulates straight into the
// caller's scale output, which is then turned into the scale in place and read
// by the fused pass -- no workspace.
template <int MODE>
rq_status dynamic_tensor_call(const void *x, const void *residual_in, void *residual_out,
                                     const void *weight, float eps, float *d_scale_out, uint8_t *q,
                                     uint8_t *sf, void *norm_out, int64_t rows, int64_t hidden,
                                     rq_dtype dt, rq_stream_t stream)
{
    const int sf_swizzled = MODE == rq::MODE_NVFP4_SWZ;
    rq_status st = check_rows(rows, hidden, dt);
    if (st != RQ_OK) return st;
    if (!d_scale_out) return RQ_ERR_NULL;
    if (!aligned4(d_scale_out)) return RQ_ERR_MISALIGNED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int nvfp4 = rq::is_nvfp4<MODE>();
    if (rows > 0) {
        if (!x || !residual_in || !residual_out || !weight || !q || (nvfp4 && !sf)) return RQ_ERR_NULL;
        if (!aligned16(x) || !aligned16(residual_in) || !aligned16(residual_out) ||
            !aligned16(weight) || !aligned16(q) || (nvfp4 && !aligned16(sf)) ||
            (norm_out && !aligned16(norm_out)))
            return RQ_ERR_MISALIGNED;
        const int64_t tb = rows * hidden * 2;
        const Span ins[] = {span(x, tb), span(residual_in, tb), span(weight, hidden * 2)};
        const Span outs[] = {span(residual_out, tb), span(norm_out, tb),
                             span(q, nvfp4 ? rows * hidden / 2 : rows * hidden),
                             span(nvfp4 ? sf : nullptr, sf_bytes(rows, hidden, sf_swizzled)),
                             span(d_scale_out, 4)};
        if (bad_alias(outs, 5, ins, 3, 0, 1)) return RQ_ERR_ALIAS;
    }
    st = cuda_status(cudaMemsetAsync(d_scale_out, 0, sizeof(float), s));
    if (st != RQ_OK) return st;
    if (rows > 0) {
        auto pa = make_params(x, residual_in, nullptr, weight, eps, nullptr, nullptr, nullptr, nullptr,
                              d_scale_out, rows, hidden);
        st = launch_rows<rq::MODE_AMAX>(pa, dt, stream);
        if (st != RQ_OK) return st;
    }
    st = cuda_status(rq::launch_scale_from_amax(d_scale_out, d_scale_out, nvfp4, 1, s));
    if (st != RQ_OK || rows == 0) return st;
    auto p = make_params(x, residual_in, residual_out, weight, eps, d_scale_out, q, sf, norm_out,
                         nullptr, rows, hidden);
    return launch_rows<MODE>(p, dt, stream);
}

rq_status nvfp4_call(const void *x, const void *residual_in, void *residual_out, const void *weight,
                     float eps, const float *d_global_scale, uint8_t *q_packed,
                     uint8_t *block_scales, void *norm_out, int64_t rows, int64_t hidden,
                     rq_dtype dt, rq_stream_t stream, int sf_swizzled)
{
    rq_status st = check_rows(rows, hidden, dt);
    if (st != RQ_OK || rows == 0) return st;
    if (!x || !residual_in || !residual_out || !weight || !d_global_scale || !q_packed ||
        !block_scales)
        return RQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(residual_in) || !aligned16(residual_out) || !aligned16(weight) ||
        !aligned16(q_packed) || !aligned16(block_scales) || (norm_out && !aligned16(norm_out)) ||
        !aligned4(d_global_scale))
        return RQ_ERR_MISALIGNED;
    const int64_t tb = rows * hidden * 2;
    const Span ins[] = {span(x, tb), span(residual_in, tb), span(weight, hidden * 2),
                        span(d_global_scale, 4)};
    const Span outs[] = {span(residual_out, tb), span(norm_out, tb), span(q_packed, rows * hidden / 2),
                         span(block_scales, sf_bytes(rows, hidden, sf_swizzled))};
    if (bad_alias(outs, 4, ins, 4, 0, 1)) return RQ_ERR_ALIAS;
    auto p = make_params(x, residual_in, residual_out, weight, eps, d_global_scale, q_packed,
                         block_scales, norm_out, nullptr, rows, hidden);
    return sf_swizzled ? launch_rows<rq::MODE_NVFP4_SWZ>(p, dt, stream)
                       : launch_rows<rq::MODE_NVFP4>(p, dt, stream);
}

}  // namespace

extern "C" {

rq_status rq_add_rmsnorm_fp8(const void *x, const void *residual_in, void *residual_out,
                             const void *weight, float eps, const float *d_scale, uint8_t *q_out,
                             void *norm_out, int64_t rows, int64_t hidden, rq_dtype dt,
                             rq_stream_t stream)
{
    rq_status st = check_rows(rows, hidden, dt);
    if (st != RQ_OK || rows == 0) return st;
    if (!x || !residual_in || !residual_out || !weight || !d_scale || !q_out) return RQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(residual_in) || !aligned16(residual_out) || !aligned16(weight) ||
        !aligned16(q_out) || (norm_out && !aligned16(norm_out)) || !aligned4(d_scale))
        return RQ_ERR_MISALIGNED;
    const int64_t tb = rows * hidden * 2;
    const Span ins[] = {span(x, tb), span(residual_in, tb), span(weight, hidden * 2), span(d_scale, 4)};
    const Span outs[] = {span(residual_out, tb), span(norm_out, tb), span(q_out, rows * hidden)};
    if (bad_alias(outs, 3, ins, 4, 0, 1)) return RQ_ERR_ALIAS;
    auto p = make_params(x, residual_in, residual_out, weight, eps, d_scale, q_out, nullptr, norm_out,
                         nullptr, rows, hidden);
    return launch_rows<rq::MODE_FP8>(p, dt, stream);
}

rq_status rq_add_rmsnorm_nvfp4(const void *x, const void *residual_in, void *residual_out,
                               const void *weight, float eps, const float *d_global_scale,
                               uint8_t *q_packed, uint8_t *block_scales, void *norm_out,
                               int64_t rows, int64_t hidden, rq_dtype dt, rq_stream_t stream)
{
    return nvfp4_call(x, residual_in, residual_out, weight, eps, d_global_scale, q_packed,
                      block_scales, norm_out, rows, hidden, dt, stream, 0);
}

rq_status rq_add_rmsnorm_nvfp4_swizzled(const void *x, const void *residual_in, void *residual_out,
                                        const void *weight, float eps, const float *d_global_scale,
                                        uint8_t *q_packed, uint8_t *block_scales, void *norm_out,
                                        int64_t rows, int64_t hidden, rq_dtype dt,
                                        rq_stream_t stream)
{
    return nvfp4_call(x, residual_in, residual_out, weight, eps, d_global_scale, q_packed,
                      block_scales, norm_out, rows, hidden, dt, stream, 1);
}

static rq_status gated_call(const void *x, const void *z, const void *weight, float eps,
                            const float *d_global_scale, uint8_t *q_packed, uint8_t *block_scales,
                            void *norm_out, int64_t rows, int64_t hidden, rq_dtype dt,
                            rq_stream_t stream, int sf_swizzled)
{
    rq_status st = check_rows(rows, hidden, dt);
    if (st != RQ_OK || rows == 0) return st;
    if (!x || !z || !weight || !d_global_scale || !q_packed || !block_scales) return RQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(z) || !aligned16(weight) || !aligned16(q_packed) ||
        !aligned16(block_scales) || (norm_out && !aligned16(norm_out)) || !aligned4(d_global_scale))
        return RQ_ERR_MISALIGNED;
    const int64_t tb = rows * hidden * 2;
    const Span ins[] = {span(x, tb), span(z, tb), span(weight, hidden * 2), span(d_global_scale, 4)};
    const Span outs[] = {span(norm_out, tb), span(q_packed, rows * hidden / 2),
                         span(block_scales, sf_bytes(rows, hidden, sf_swizzled))};
    if (bad_alias(outs, 3, ins, 4)) return RQ_ERR_ALIAS;
    auto p = make_params(x, z, nullptr, weight, eps, d_global_scale, q_packed, block_scales,
                         norm_out, nullptr, rows, hidden);
    return sf_swizzled ? launch_rows<rq::MODE_GATED_NVFP4_SWZ>(p, dt, stream)
                       : launch_rows<rq::MODE_GATED_NVFP4>(p, dt, stream);
}

rq_status rq_gated_rmsnorm_nvfp4(const void *x, const void *z, const void *weight, float eps,
                                 const float *d_global_scale, uint8_t *q_packed,
                                 uint8_t *block_scales, void *norm_out, int64_t rows,
                                 int64_t hidden, rq_dtype dt, rq_stream_t stream)
{
    return gated_call(x, z, weight, eps, d_global_scale, q_packed, block_scales, norm_out, rows,
                      hidden, dt, stream, 0);
}

rq_status rq_gated_rmsnorm_nvfp4_swizzled(const void *x, const void *z, const void *weight,
                                          float eps, const float *d_global_scale,
                                          uint8_t *q_packed, uint8_t *block_scales,
                                          void *norm_out, int64_t rows, int64_t hidden,
                                          rq_dtype dt, rq_stream_t stream)
{
    return gated_call(x, z, weight, eps, d_global_scale, q_packed, block_scales, norm_out, rows,
                      hidden, dt, stream, 1);
}

rq_status rq_add_rmsnorm_amax(const void *x, const void *residual_in, const void *weight, float eps,
                              float *d_amax, int64_t rows, int64_t hidden, rq_dtype dt,
                              rq_stream_t stream)
{
    rq_status st = check_rows(rows, hidden, dt);
    if (st != RQ_OK) return st;
    if (!d_amax) return RQ_ERR_NULL;
    if (rows > 0 && (!x || !residual_in || !weight)) return RQ_ERR_NULL;
    if (!aligned4(d_amax) || (rows > 0 && (!aligned16(x) || !aligned16(residual_in) ||
                                            !aligned16(weight))))
        return RQ_ERR_MISALIGNED;
    const int64_t tb = rows * hidden * 2;
    const Span ins[] = {span(x, tb), span(residual_in, tb), span(weight, hidden * 2)};
    const Span outs[] = {span(d_amax, 4)};
    if (bad_alias(outs, 1, ins, 3)) return RQ_ERR_ALIAS;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    st = cuda_status(cudaMemsetAsync(d_amax, 0, sizeof(float), s));
    if (st != RQ_OK || rows == 0) return st;
    auto p = make_params(x, residual_in, nullptr, weight, eps, nullptr, nullptr, nullptr, nullptr,
                         d_amax, rows, hidden);
    return launch_rows<rq::MODE_AMAX>(p, dt, stream);
}

static rq_status scale_from_amax(const float *d_amax, float *d_out, int nvfp4, rq_stream_t stream)
{
    if (!d_amax || !d_out) return RQ_ERR_NULL;
    if (!aligned4(d_amax) || !aligned4(d_out)) return RQ_ERR_MISALIGNED;
    return cuda_status(
        rq::launch_scale_from_amax(d_amax, d_out, nvfp4, 0, reinterpret_cast<cudaStream_t>(stream)));
}

rq_status rq_fp8_scale_from_amax(const float *d_amax, float *d_scale, rq_stream_t stream)
{
    return scale_from_amax(d_amax, d_scale, 0, stream);
}

rq_status rq_nvfp4_global_scale_from_amax(const float *d_amax, float *d_gs, rq_stream_t stream)
{
    return scale_from_amax(d_amax, d_gs, 1, stream);
}

rq_status rq_add_rmsnorm_fp8_per_token(const void *x, const void *residual_in, void *residual_out,
                                       const void *weight, float eps, uint8_t *q_out,
                                       float *d_row_scales, void *norm_out, int64_t rows,
                                       int64_t hidden, rq_dtype dt, rq_stream_t stream)
{
    rq_status st = check_rows(rows, hidden, dt);
    if (st != RQ_OK || rows == 0) return st;
    if (!x || !residual_in || !residual_out || !weight || !q_out || !d_row_scales) return RQ_ERR_NULL;
    if (!aligned16(x) || !aligned16(residual_in) || !aligned16(residual_out) || !aligned16(weight) ||
        !aligned16(q_out) || (norm_out && !aligned16(norm_out)) || !aligned4(d_row_scales))
        return RQ_ERR_MISALIGNED;
    const int64_t tb = rows * hidden * 2;
    const Span ins[] = {span(x, tb), span(residual_in, tb), span(weight, hidden * 2)};
    const Span outs[] = {span(residual_out, tb), span(norm_out, tb), span(q_out, rows * hidden),
                         span(d_row_scales, rows * 4)};
    if (bad_alias(outs, 4, ins, 3, 0, 1)) return RQ_ERR_ALIAS;
    auto p = make_params(x, residual_in, residual_out, weight, eps, nullptr, q_out, nullptr, norm_out,
                         nullptr, rows, hidden);
    p.row_scales = d_row_scales;
    return launch_rows<rq::MODE_FP8_ROW>(p, dt, stream);
}

rq_status rq_add_rmsnorm_fp8_dynamic(const void *x, const void *residual_in, void *residual_out,
                                     const void *weight, float eps, float *d_scale_out,
                                     uint8_t *q_out, void *norm_out, int64_t rows, int64_t hidden,
                                     rq_dtype dt, rq_stream_t stream)
{
    return dynamic_tensor_call<rq::MODE_FP8>(x, residual_in, residual_out, weight, eps, d_scale_out,
                                             q_out, nullptr, norm_out, rows, hidden, dt, stream);
}

rq_status rq_add_rmsnorm_nvfp4_dynamic(const void *x, const void *residual_in, void *residual_out,
                                       const void *weight, float eps, float *d_global_scale_out,
                                       uint8_t *q_packed, uint8_t *block_scales, void *norm_out,
                                       int64_t rows, int64_t hidden, rq_dtype dt,
                                       rq_stream_t stream)
{
    return dynamic_tensor_call<rq::MODE_NVFP4>(x, residual_in, residual_out, weight, eps,
                                               d_global_scale_out, q_packed, block_scales, norm_out,
                                               rows, hidden, dt, stream);
}

rq_status rq_add_rmsnorm_nvfp4_dynamic_swizzled(const void *x, const void *residual_in,
                                                void *residual_out, const void *weight, float eps,
                                                float *d_global_scale_out, uint8_t *q_packed,
                                                uint8_t *block_scales, void *norm_out,
                                                int64_t rows, int64_t hidden, rq_dtype dt,
                                                rq_stream_t stream)
{
    return dynamic_tensor_call<rq::MODE_NVFP4_SWZ>(x, residual_in, residual_out, weight, eps,
                                               d_global_scale_out, q_packed, block_scales, norm_out,
                                               rows, hidden, dt, stream);
}

}  // extern "C"

namespace {

// What a Q/K entry point asks of the kernel beyond the common arguments.
struct QKCall {
    int mode = rq::QK_STORE;
    int rope_dim = RQ_QK_HEAD_DIM;       // QK_MIXED: the rotated tail of each head
    const int64_t *k_slots = nullptr;    // KV-pool calls
    int64_t num_slots = 0;
    float *q_amax = nullptr, *k_amax = nullptr;  // QK_AMAX
};

// Argument checks of every Q/K call, then the launch.
rq_status qk_call(const void *q, const void *k, int64_t q_token_stride, int64_t k_token_stride,
                  int64_t n_tokens, int n_q_heads, int n_k_heads, int head_dim,
                  const void *q_weight, const void *k_weight, float eps, const int32_t *positions,
                  const float *cos_sin_cache, int64_t max_pos, const float *d_q_scale,
                  const float *d_k_scale, uint8_t *q_out, uint8_t *k_out, const QKCall &c,
                  rq_dtype dt, rq_stream_t stream)
{
    const bool amax = c.mode == rq::QK_AMAX, mixed = c.mode == rq::QK_MIXED;
    if (dt != RQ_BF16 && dt != RQ_FP16) return RQ_ERR_DTYPE;
    // limits that keep every byte extent below 2^63 and the head count in an int
    if (n_tokens < 0 || n_q_heads < 0 || n_k_heads < 0 || max_pos < 1 || n_tokens > (int64_t)1 << 36 ||
        n_q_heads > RQ_QK_MAX_HEADS || n_k_heads > RQ_QK_MAX_HEADS || max_pos > (int64_t)1 << 40 ||
        q_token_stride > (int64_t)1 << 40 || k_token_stride > (int64_t)1 << 40 ||
        (c.k_slots && c.num_slots > (int64_t)1 << 40))
        return RQ_ERR_SHAPE;
    if (head_dim != RQ_QK_HEAD_DIM) return RQ_ERR_UNSUPPORTED;
    if (mixed && c.rope_dim != 16 && c.rope_dim != 32 && c.rope_dim != 64 && c.rope_dim != 128)
        return RQ_ERR_UNSUPPORTED;
    if (n_tokens == 0 || (n_q_heads == 0 && n_k_heads == 0)) return RQ_OK;
    const bool has_q = n_q_heads > 0, has_k = n_k_heads > 0;
    if (has_q && (q_token_stride < (int64_t)n_q_heads * head_dim || q_token_stride % 8 != 0))
        return q_token_stride % 8 != 0 ? RQ_ERR_MISALIGNED : RQ_ERR_SHAPE;
    if (has_k && (k_token_stride < (int64_t)n_k_heads * head_dim || k_token_stride % 8 != 0))
        return k_token_stride % 8 != 0 ? RQ_ERR_MISALIGNED : RQ_ERR_SHAPE;
    if (!positions || !cos_sin_cache) return RQ_ERR_NULL;
    if (has_q && (!q || !q_weight || (!amax && (!d_q_scale || !q_out)) || (amax && !c.q_amax)))
        return RQ_ERR_NULL;
    if (has_k && (!k || !k_weight || (!amax && (!d_k_scale || !k_out)) || (amax && !c.k_amax)))
        return RQ_ERR_NULL;
    if (c.k_slots && has_k && c.num_slots < 0) return RQ_ERR_SHAPE;
    if (!aligned16(cos_sin_cache) || !aligned4(positions) ||
        (c.k_slots && (reinterpret_cast<uintptr_t>(c.k_slots) & 7u)))
        return RQ_ERR_MISALIGNED;
    if (has_q && (!aligned16(q) || !aligned16(q_weight) ||
                  (!amax && (!aligned16(q_out) || !aligned4(d_q_scale))) ||
                  (amax && !aligned4(c.q_amax))))
        return RQ_ERR_MISALIGNED;
    if (has_k && (!aligned16(k) || !aligned16(k_weight) ||
                  (!amax && (!aligned16(k_out) || !aligned4(d_k_scale))) ||
                  (amax && !aligned4(c.k_amax))))
        return RQ_ERR_MISALIGNED;
    // input extents: the last token's heads end before (T-1)*stride + H*D
    const int64_t qin = has_q ? ((n_tokens - 1) * q_token_stride + (int64_t)n_q_heads * head_dim) * 2 : 0;
    const int64_t kin = has_k ? ((n_tokens - 1) * k_token_stride + (int64_t)n_k_heads * head_dim) * 2 : 0;
    const int64_t table_cols = mixed ? c.rope_dim : head_dim;
    const int64_t k_rows = c.k_slots ? c.num_slots : n_tokens;
    const int64_t k_head_bytes = mixed ? head_dim + c.rope_dim : head_dim;
    const Span ins[] = {span(has_q ? q : nullptr, qin), span(has_k ? k : nullptr, kin),
                        span(has_q ? q_weight : nullptr, head_dim * 2),
                        span(has_k ? k_weight : nullptr, head_dim * 2), span(positions, n_tokens * 4),
                        span(cos_sin_cache, max_pos * table_cols * 4),
                        span(has_q && !amax ? d_q_scale : nullptr, 4),
                        span(has_k && !amax ? d_k_scale : nullptr, 4),
                        span(has_k ? c.k_slots : nullptr, n_tokens * 8)};
    if (amax) {
        // the two maxima may share one address (one maximum over Q and K)
        const Span qa = span(has_q ? c.q_amax : nullptr, 4), ka = span(has_k ? c.k_amax : nullptr, 4);
        if (bad_alias(&qa, 1, ins, 9) || bad_alias(&ka, 1, ins, 9)) return RQ_ERR_ALIAS;
    } else {
        const Span outs[] = {span(has_q ? q_out : nullptr, n_tokens * n_q_heads * (int64_t)head_dim),
                             span(has_k ? k_out : nullptr, k_rows * n_k_heads * k_head_bytes)};
        if (bad_alias(outs, 2, ins, 9)) return RQ_ERR_ALIAS;
    }

    rq::QKParams p;
    p.q = q;
    p.k = k;
    p.q_stride = q_token_stride;
    p.k_stride = k_token_stride;
    p.n_tokens = n_tokens;
    p.hq = n_q_heads;
    p.hk = n_k_heads;
    p.qw = q_weight;
    p.kw = k_weight;
    p.eps = eps;
    p.pos = positions;
    p.cos_sin = cos_sin_cache;
    p.max_pos = max_pos;
    p.q_scale = d_q_scale;
    p.k_scale = d_k_scale;
    p.q_out = q_out;
    p.k_out = k_out;
    p.k_slots = has_k ? c.k_slots : nullptr;
    p.num_slots = c.num_slots;
    p.rope_dim = mixed ? c.rope_dim : head_dim;
    p.q_amax = c.q_amax;
    p.k_amax = c.k_amax;
    p.nz = -0.0f;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (amax) {
        cudaError_t e = cudaSuccess;
        if (has_q) e = cudaMemsetAsync(c.q_amax, 0, sizeof(float), s);
        if (e == cudaSuccess && has_k) e = cudaMemsetAsync(c.k_amax, 0, sizeof(float), s);
        if (e != cudaSuccess) return cuda_status(e);
    }
    cudaError_t e;
    if (c.mode == rq::QK_AMAX)
        e = dt == RQ_BF16 ? rq::launch_qk_rmsnorm_rope<rq::BF16, rq::QK_AMAX>(p, s)
                          : rq::launch_qk_rmsnorm_rope<rq::FP16, rq::QK_AMAX>(p, s);
    else if (c.mode == rq::QK_MIXED)
        e = dt == RQ_BF16 ? rq::launch_qk_rmsnorm_rope<rq::BF16, rq::QK_MIXED>(p, s)
                          : rq::launch_qk_rmsnorm_rope<rq::FP16, rq::QK_MIXED>(p, s);
    else
        e = dt == RQ_BF16 ? rq::launch_qk_rmsnorm_rope<rq::BF16, rq::QK_STORE>(p, s)
                          : rq::launch_qk_rmsnorm_rope<rq::FP16, rq::QK_STORE>(p, s);
    return cuda_status(e);
}

}  // namespace

extern "C" {

rq_status rq_qk_rmsnorm_rope_fp8(const void *q, const void *k, int64_t q_token_stride,
                                 int64_t k_token_stride, int64_t n_tokens, int n_q_heads,
                                 int n_k_heads, int head_dim, const void *q_weight,
                                 const void *k_weight, float eps, const int32_t *positions,
                                 const float *cos_sin_cache, int64_t max_pos,
                                 const float *d_q_scale, const float *d_k_scale, uint8_t *q_out,
                                 uint8_t *k_out, rq_dtype dt, rq_stream_t stream)
{
    return qk_call(q, k, q_token_stride, k_token_stride, n_tokens, n_q_heads, n_k_heads, head_dim,
                   q_weight, k_weight, eps, positions, cos_sin_cache, max_pos, d_q_scale, d_k_scale,
                   q_out, k_out, QKCall{}, dt, stream);
}

rq_status rq_qk_rmsnorm_rope_fp8_kv_store(const void *q, const void *k, int64_t q_token_stride,
                                          int64_t k_token_stride, int64_t n_tokens, int n_q_heads,
                                          int n_k_heads, int head_dim, const void *q_weight,
                                          const void *k_weight, float eps,
                                          const int32_t *positions, const float *cos_sin_cache,
                                          int64_t max_pos, const float *d_q_scale,
                                          const float *d_k_scale, uint8_t *q_out,
                                          uint8_t *k_pool, const int64_t *k_slots,
                                          int64_t num_slots, rq_dtype dt, rq_stream_t stream)
{
    if (n_k_heads > 0 && n_tokens > 0 && !k_slots) return RQ_ERR_NULL;
    QKCall c;
    c.k_slots = k_slots;
    c.num_slots = num_slots;
    return qk_call(q, k, q_token_stride, k_token_stride, n_tokens, n_q_heads, n_k_heads, head_dim,
                   q_weight, k_weight, eps, positions, cos_sin_cache, max_pos, d_q_scale, d_k_scale,
                   q_out, k_pool, c, dt, stream);
}

rq_status rq_qk_rmsnorm_rope_fp8_kv_store_mixed(
    const void *q, const void *k, int64_t q_token_stride, int64_t k_token_stride, int64_t n_tokens,
    int n_q_heads, int n_k_heads, int head_dim, int rope_dim, const void *q_weight,
    const void *k_weight, float eps, const int32_t *positions, const float *cos_sin_cache,
    int64_t max_pos, const float *d_q_scale, const float *d_k_scale, uint8_t *q_out,
    uint8_t *k_pool, const int64_t *k_slots, int64_t num_slots, rq_dtype dt, rq_stream_t stream)
{
    if (n_k_heads > 0 && n_tokens > 0 && !k_slots) return RQ_ERR_NULL;
    QKCall c;
    c.mode = rq::QK_MIXED;
    c.rope_dim = rope_dim;
    c.k_slots = k_slots;
    c.num_slots = num_slots;
    return qk_call(q, k, q_token_stride, k_token_stride, n_tokens, n_q_heads, n_k_heads, head_dim,
                   q_weight, k_weight, eps, positions, cos_sin_cache, max_pos, d_q_scale, d_k_scale,
                   q_out, k_pool, c, dt, stream);
}

rq_status rq_qk_rmsnorm_rope_amax(const void *q, const void *k, int64_t q_token_stride,
                                  int64_t k_token_stride, int64_t n_tokens, int n_q_heads,
                                  int n_k_heads, int head_dim, const void *q_weight,
                                  const void *k_weight, float eps, const int32_t *positions,
                                  const float *cos_sin_cache, int64_t max_pos, float *d_q_amax,
                                  float *d_k_amax, rq_dtype dt, rq_stream_t stream)
{
    QKCall c;
    c.mode = rq::QK_AMAX;
    c.q_amax = d_q_amax;
    c.k_amax = d_k_amax;
    rq_status st = qk_call(q, k, q_token_stride, k_token_stride, n_tokens, n_q_heads, n_k_heads,
                           head_dim, q_weight, k_weight, eps, positions, cos_sin_cache, max_pos,
                           nullptr, nullptr, nullptr, nullptr, c, dt, stream);
    if (st != RQ_OK || (n_tokens > 0 && (n_q_heads > 0 || n_k_heads > 0))) return st;
    // an empty call still clears the maxima it was given
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n_q_heads > 0 && d_q_amax) {
        if (!aligned4(d_q_amax)) return RQ_ERR_MISALIGNED;
        st = cuda_status(cudaMemsetAsync(d_q_amax, 0, sizeof(float), s));
    }
    if (st == RQ_OK && n_k_heads > 0 && d_k_amax) {
        if (!aligned4(d_k_amax)) return RQ_ERR_MISALIGNED;
        st = cuda_status(cudaMemsetAsync(d_k_amax, 0, sizeof(float), s));
    }
    return st;
}

rq_status rq_qk_rmsnorm_rope_fp8_dynamic(const void *q, const void *k, int64_t q_token_stride,
                                         int64_t k_token_stride, int64_t n_tokens, int n_q_heads,
                                         int n_k_heads, int head_dim, const void *q_weight,
                                         const void *k_weight, float eps,
                                         const int32_t *positions, const float *cos_sin_cache,
                                         int64_t max_pos, float *d_q_scale_out,
                                         float *d_k_scale_out, uint8_t *q_out, uint8_t *k_out,
                                         rq_dtype dt, rq_stream_t stream)
{
    // the maxima accumulate in the caller's scale outputs, which the fused
    // pass then reads: no workspace
    rq_status st = rq_qk_rmsnorm_rope_amax(q, k, q_token_stride, k_token_stride, n_tokens,
                                           n_q_heads, n_k_heads, head_dim, q_weight, k_weight, eps,
                                           positions, cos_sin_cache, max_pos, d_q_scale_out,
                                           d_k_scale_out, dt, stream);
    if (st != RQ_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n_q_heads > 0 && d_q_scale_out)
        st = cuda_status(rq::launch_scale_from_amax(d_q_scale_out, d_q_scale_out, 0, 1, s));
    if (st == RQ_OK && n_k_heads > 0 && d_k_scale_out && d_k_scale_out != d_q_scale_out)
        st = cuda_status(rq::launch_scale_from_amax(d_k_scale_out, d_k_scale_out, 0, 1, s));
    if (st != RQ_OK || n_tokens == 0) return st;
    return qk_call(q, k, q_token_stride, k_token_stride, n_tokens, n_q_heads, n_k_heads, head_dim,
                   q_weight, k_weight, eps, positions, cos_sin_cache, max_pos, d_q_scale_out,
                   d_k_scale_out, q_out, k_out, QKCall{}, dt, stream);
}

size_t rq_nvfp4_packed_bytes(int64_t rows, int64_t hidden)
{
    return rows > 0 && hidden > 0 ? (size_t)rows * (size_t)hidden / 2 : 0;
}

size_t rq_nvfp4_scale_bytes(int64_t rows, int64_t hidden)
{
    return rows > 0 && hidden > 0 ? (size_t)sf_bytes(rows, hidden, 0) : 0;
}

size_t rq_nvfp4_swizzled_scale_bytes(int64_t rows, int64_t hidden)
{
    return rows > 0 && hidden > 0 ? (size_t)sf_bytes(rows, hidden, 1) : 0;
}

const char *rq_status_string(rq_status status)
{
    switch (status) {
    case RQ_OK: return "RQ_OK";
    case RQ_ERR_NULL: return "RQ_ERR_NULL: a required pointer is NULL";
    case RQ_ERR_SHAPE: return "RQ_ERR_SHAPE: invalid rows, hidden, stride or head count";
    case RQ_ERR_DTYPE: return "RQ_ERR_DTYPE: dtype must be RQ_BF16 or RQ_FP16";
    case RQ_ERR_MISALIGNED: return "RQ_ERR_MISALIGNED: tensors need 16-byte alignment, scalars 4";
    case RQ_ERR_ALIAS: return "RQ_ERR_ALIAS: an output overlaps another argument";
    case RQ_ERR_UNSUPPORTED: return "RQ_ERR_UNSUPPORTED: hidden above the maximum or head_dim != 128";
    case RQ_ERR_CUDA: return "RQ_ERR_CUDA: the CUDA runtime reported an error";
    }
    return "unknown rq_status";
}

const char *rq_last_error(void) { return g_last_error; }

int rq_version(void) { return 200; }

}  // extern "C"
