/*
 * rq.h -- C ABI of librq: fused residual add + RMSNorm + FP8 / NVFP4
 * quantisation, and per-head Q/K RMSNorm + RoPE + FP8 store, for NVIDIA
 * GB300 (sm_103a).
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller, row-major
 *    and contiguous unless a stride argument says otherwise.  The library
 *    allocates no device memory and keeps no state besides a per-device cache
 *    of launch limits.
 *  - Scales are fp32 scalars in device memory, read by the kernel, so a call
 *    never synchronises with the host.
 *  - Work is enqueued on `stream` (NULL = the legacy default stream) and is
 *    asynchronous: a returned RQ_OK means the launch was accepted.  Kernels
 *    are launched with programmatic stream serialisation: their thread
 *    blocks may be scheduled while the previous kernel in the stream is
 *    finishing, and wait for it to complete before their first memory
 *    access, so stream order holds as for a plain launch (also under graph
 *    capture, where the dependency is a programmatic edge).
 *  - Every argument check runs on the host before any CUDA call; a failed
 *    check returns an error status and launches nothing.  Nothing throws
 *    across the ABI.  A call with rows == 0 (or n_tokens == 0) returns RQ_OK
 *    once its dtype and shape arguments are valid, whatever its pointers
 *    (empty tensors may have NULL data), and launches nothing.
 *  - Alignment: every tensor pointer must be 16-byte aligned; scalar pointers
 *    4-byte aligned.
 *  - Aliasing: residual_out may equal residual_in exactly (in-place residual
 *    update); any other overlap between an output and another argument
 *    returns RQ_ERR_ALIAS.
 *
 * Numerics (every fp32 step is one IEEE round-to-nearest-even operation; the
 * only freedom is the order of the fp32 sum of squares):
 *   s_i  = dt(x_i + r_i)                                   (residual')
 *   rstd = 1 / sqrt(sum_i s_i^2 / hidden + eps)
 *   y_i  = dt((s_i * rstd) * w_i)                          (norm output)
 *   FP8:   q_i = E4M3(y_i / scale)           round to nearest even, satfinite
 *   NVFP4: per 16-element block, a = max |y_i|,
 *          sf = E4M3((gs * a) / 6), enc = gs / sf (0 if sf == 0),
 *          c_i = E2M1(y_i * enc), packed two per byte, even element in the
 *          low nibble; dequantised value = e2m1(c_i) * sf / gs.
 */
#ifndef RQ_H
#define RQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; declared here so that the header needs no
 * CUDA include. */
struct CUstream_st;
typedef struct CUstream_st *rq_stream_t;

typedef enum {
    RQ_OK = 0,
    RQ_ERR_NULL = 1,        /* a required pointer is NULL */
    RQ_ERR_SHAPE = 2,       /* rows < 0, hidden <= 0 or % 16 != 0, bad stride ... */
    RQ_ERR_DTYPE = 3,       /* dtype is neither RQ_BF16 nor RQ_FP16 */
    RQ_ERR_MISALIGNED = 4,  /* a pointer or stride breaks the 16-byte rule */
    RQ_ERR_ALIAS = 5,       /* an output overlaps another argument */
    RQ_ERR_UNSUPPORTED = 6, /* hidden > RQ_MAX_HIDDEN, head_dim != 128 ... */
    RQ_ERR_CUDA = 7         /* the CUDA runtime refused the launch; see rq_last_error() */
} rq_status;

/* Storage type of x, residual, weight and norm_out (all must match). */
typedef enum { RQ_BF16 = 0, RQ_FP16 = 1 } rq_dtype;

#define RQ_MAX_HIDDEN 262144
#define RQ_QK_HEAD_DIM 128
#define RQ_QK_MAX_HEADS 65536

/*
 * Residual add + RMSNorm + per-tensor FP8 E4M3.
 * Source: "Add NanoJet backend for AutoDeploy prefill-only FP8 inference"
 * (TensorRT-LLM PR 17288), Description: RMSNorm with FP8 quantisation in the
 * kernel epilogue; residual add folded in place (same page, Test Coverage:
 * residual folding with aliasing).
 *
 *   x, residual_in      [rows, hidden] dt, read
 *   residual_out        [rows, hidden] dt, written with s (may == residual_in)
 *   weight              [hidden] dt
 *   d_scale             device fp32 dequant scale (q = y / scale)
 *   q_out               [rows, hidden] E4M3 bytes
 *   norm_out            [rows, hidden] dt, written with y; may be NULL
 *   hidden              multiple of 16, <= RQ_MAX_HIDDEN
 */
rq_status rq_add_rmsnorm_fp8(const void *x, const void *residual_in,
                             void *residual_out, const void *weight,
                             float eps, const float *d_scale, uint8_t *q_out,
                             void *norm_out, int64_t rows, int64_t hidden,
                             rq_dtype dt, rq_stream_t stream);

/*
 * Residual add + RMSNorm (+ high-precision norm output) + NVFP4.
 * Source: "Add AutoDeploy NVFP4 RMSNorm quant fusion" (TensorRT-LLM PR 14361),
 * Changes: fused add + RMSNorm + NVFP4 ops with and without the norm output;
 * "[Performance]: Fuse local NVFP4 tail after NCCL fallback" (TensorRT-LLM
 * issue 17900), Proposal: the one-launch residual + RMSNorm + NVFP4 tail and
 * its support conditions (FP16/BF16 contiguous matching dtypes, FP32 scalar
 * per-tensor scale, no bias, hidden % 16 == 0).
 *
 *   d_global_scale      device fp32 gs in the quantising direction (e.g.
 *                       448 * 6 / amax(y))
 *   q_packed            [rows, hidden / 2] bytes (rq_nvfp4_packed_bytes)
 *   block_scales        [rows, hidden / 16] E4M3 bytes, row-major
 *                       (rq_nvfp4_scale_bytes)
 *   other arguments as in rq_add_rmsnorm_fp8
 */
rq_status rq_add_rmsnorm_nvfp4(const void *x, const void *residual_in,
                               void *residual_out, const void *weight,
                               float eps, const float *d_global_scale,
                               uint8_t *q_packed, uint8_t *block_scales,
                               void *norm_out, int64_t rows, int64_t hidden,
                               rq_dtype dt, rq_stream_t stream);

/*
 * Per-head Q/K RMSNorm + NeoX RoPE + uniform FP8 E4M3 store.
 * Source: "Add NanoJet backend for AutoDeploy prefill-only FP8 inference",
 * Description (fused Q/K RMSNorm and RoPE); "perf: add fused norm + RoPE +
 * uniform fp8 store for TRT-LLM DSv4 sparse attention" (SGLang PR 32975),
 * review thread (norm, RoPE and a uniform FP8 store in one kernel).
 *
 *   q, k                token t, head h starts at q + t*q_token_stride +
 *                       h*head_dim elements (strides in elements, multiples
 *                       of 8, >= n_heads*head_dim); heads are contiguous
 *   q_weight, k_weight  [head_dim] dt, shared by all heads of Q (resp. K)
 *   positions           [n_tokens] int32; values outside [0, max_pos) are
 *                       clamped into it
 *   cos_sin_cache       [max_pos, head_dim] fp32: cos of the head_dim/2
 *                       frequencies, then their sin
 *   d_q_scale, d_k_scale device fp32 dequant scales (may be the same pointer)
 *   q_out, k_out        [n_tokens, n_*_heads, head_dim] E4M3 bytes (dense)
 *   head_dim            must be RQ_QK_HEAD_DIM (128)
 *   n_q_heads or n_k_heads may be 0, in which case that side's pointers may
 *   be NULL.
 * Limits (RQ_ERR_SHAPE beyond them): n_tokens <= 2^36, heads per side <=
 * RQ_QK_MAX_HEADS, max_pos, token strides and num_slots <= 2^40.
 * Per head: n = dt(RMSNorm(x) * w); o_i = dt(n_i c_i - n_{i+64} s_i),
 * o_{i+64} = dt(n_{i+64} c_i + n_i s_i); out = E4M3(o / scale).
 */
rq_status rq_qk_rmsnorm_rope_fp8(const void *q, const void *k,
                                 int64_t q_token_stride,
                                 int64_t k_token_stride, int64_t n_tokens,
                                 int n_q_heads, int n_k_heads, int head_dim,
                                 const void *q_weight, const void *k_weight,
                                 float eps, const int32_t *positions,
                                 const float *cos_sin_cache, int64_t max_pos,
                                 const float *d_q_scale,
                                 const float *d_k_scale, uint8_t *q_out,
                                 uint8_t *k_out, rq_dtype dt,
                                 rq_stream_t stream);

/*
 * The same Q/K call with K's codes stored into a KV-cache pool instead of a
 * dense tensor: token t's K heads go to pool row k_slots[t] of
 * k_pool[num_slots, n_k_heads, head_dim] (E4M3 bytes).  A slot outside
 * [0, num_slots) (e.g. -1 for a padding token) stores nothing for that
 * token.  Q is written densely to q_out as above.
 * Source: "perf: add fused norm + RoPE + uniform fp8 store for TRT-LLM DSv4
 * sparse attention" (SGLang PR 32975), review thread: the norm + RoPE kernel
 * with a store epilogue into a uniform FP8 KV pool.
 *   k_slots   [n_tokens] int64 (8-byte aligned); required when n_k_heads > 0.
 *             Two tokens with the same slot both write that pool row; which
 *             one lands last is unspecified, so slots should be distinct.
 */
rq_status rq_qk_rmsnorm_rope_fp8_kv_store(
    const void *q, const void *k, int64_t q_token_stride,
    int64_t k_token_stride, int64_t n_tokens, int n_q_heads, int n_k_heads,
    int head_dim, const void *q_weight, const void *k_weight, float eps,
    const int32_t *positions, const float *cos_sin_cache, int64_t max_pos,
    const float *d_q_scale, const float *d_k_scale, uint8_t *q_out,
    uint8_t *k_pool, const int64_t *k_slots, int64_t num_slots, rq_dtype dt,
    rq_stream_t stream);

/*
 * The Q/K call with K stored into a mixed KV-cache pool: FP8 for the part of
 * each head that RoPE leaves alone ("nope") and the dtype for the rotated
 * part ("rope").  Each head of 128 elements is read as [nope | rope] with the
 * rotated part its LAST rope_dim elements:
 *   n   = dt(RMSNorm(x) * w) over the whole head, as in the other Q/K calls;
 *   NeoX RoPE on the last rope_dim elements only, pairs (j, j + rope_dim/2)
 *   with j = 128 - rope_dim + i, i < rope_dim/2, angles cos_sin_cache[pos][i]
 *   and cos_sin_cache[pos][rope_dim/2 + i]; the first 128 - rope_dim
 *   elements pass unchanged (o = n);
 *   Q: out = E4M3(o / q_scale) for all 128 elements, dense in q_out;
 *   K: pool row k_slots[t], per head 128 + rope_dim bytes: the E4M3 codes
 *      E4M3(o / k_scale) of the first 128 - rope_dim elements, then the last
 *      rope_dim elements o as dtype values (2 bytes each, little-endian).
 * Source: "perf: add fused norm + RoPE + uniform fp8 store for TRT-LLM DSv4
 * sparse attention" (SGLang PR 32975), review thread: the FlashMLA
 * counterpart's fused store into an "fp8 nope + bf16 rope" KV pool.  The
 * page does not give the split of a head; the one above is a reading (the
 * rotated part last, one per-tensor scale for the FP8 part).
 *   rope_dim       16, 32, 64 or 128 (else RQ_ERR_UNSUPPORTED)
 *   cos_sin_cache  [max_pos, rope_dim] fp32: rope_dim/2 cos, then rope_dim/2 sin
 *   k_pool         [num_slots, n_k_heads, 128 + rope_dim] bytes (16-byte
 *                  aligned); a slot outside [0, num_slots) stores nothing
 *   k_slots        [n_tokens] int64 (8-byte aligned); required when
 *                  n_k_heads > 0.  Two tokens with the same slot both write
 *                  that row; which one lands last is unspecified.
 *   other arguments as in rq_qk_rmsnorm_rope_fp8.
 */
rq_status rq_qk_rmsnorm_rope_fp8_kv_store_mixed(
    const void *q, const void *k, int64_t q_token_stride,
    int64_t k_token_stride, int64_t n_tokens, int n_q_heads, int n_k_heads,
    int head_dim, int rope_dim, const void *q_weight, const void *k_weight,
    float eps, const int32_t *positions, const float *cos_sin_cache,
    int64_t max_pos, const float *d_q_scale, const float *d_k_scale,
    uint8_t *q_out, uint8_t *k_pool, const int64_t *k_slots, int64_t num_slots,
    rq_dtype dt, rq_stream_t stream);

/*
 * Q/K calibration: *d_q_amax = max |o| over every element of Q and *d_k_amax
 * = max |o| over K, o the dtype-rounded output of the Q/K RMSNorm + RoPE (the
 * values rq_qk_rmsnorm_rope_fp8 quantises).  Nothing else is written.  The
 * call clears both on `stream` first; they may be the same address, which
 * then receives one maximum over Q and K.  A side with no heads leaves its
 * pointer untouched (it may be NULL).
 * Source: the per-tensor scales of the pages are absolute maxima of the
 * tensor they scale ("Add AutoDeploy NVFP4 RMSNorm quant fusion", Changes:
 * reference module with input-scale calibration); for Q and K that tensor is
 * the rotated output, one scale each.
 */
rq_status rq_qk_rmsnorm_rope_amax(const void *q, const void *k,
                                  int64_t q_token_stride,
                                  int64_t k_token_stride, int64_t n_tokens,
                                  int n_q_heads, int n_k_heads, int head_dim,
                                  const void *q_weight, const void *k_weight,
                                  float eps, const int32_t *positions,
                                  const float *cos_sin_cache, int64_t max_pos,
                                  float *d_q_amax, float *d_k_amax,
                                  rq_dtype dt, rq_stream_t stream);

/*
 * The Q/K call with dynamic per-tensor scales: the amax pass above
 * accumulates into d_q_scale_out / d_k_scale_out, which are turned in place
 * into the dequant scales amax / 448 (1 for a zero maximum), and the fused
 * pass of rq_qk_rmsnorm_rope_fp8 then reads them.  No workspace.  The two
 * outputs may be the same address (one scale for Q and K).
 * Source: as rq_qk_rmsnorm_rope_amax.
 */
rq_status rq_qk_rmsnorm_rope_fp8_dynamic(
    const void *q, const void *k, int64_t q_token_stride,
    int64_t k_token_stride, int64_t n_tokens, int n_q_heads, int n_k_heads,
    int head_dim, const void *q_weight, const void *k_weight, float eps,
    const int32_t *positions, const float *cos_sin_cache, int64_t max_pos,
    float *d_q_scale_out, float *d_k_scale_out, uint8_t *q_out, uint8_t *k_out,
    rq_dtype dt, rq_stream_t stream);

/*
 * Gated RMSNorm + NVFP4: the NVFP4 call with the residual add replaced by a
 * SiLU gate applied before the norm, and nothing written back:
 *   g_i = dt(x_i * dt(silu(z_i))),  silu(z) = z / (1 + e^-z)
 *   y_i = dt((g_i * rstd) * w_i),   rstd = 1 / sqrt(sum_i g_i^2 / hidden + eps)
 * then the NVFP4 steps of rq_add_rmsnorm_nvfp4 on y (linear block scales).
 * Source: "Add AutoDeploy NVFP4 RMSNorm quant fusion", Changes: the fused
 * gated RMSNorm + NVFP4 op.  The page does not give the gating formula; the
 * one above is the separated sequence such an op replaces (gate, then the
 * norm over the whole row).  dt(silu(z)) is exact: silu(z) rounded once to
 * fp32, then to the dtype, for every finite dtype value z.
 *   x, z          [rows, hidden] dt, read
 *   norm_out      [rows, hidden] dt, written with y; may be NULL
 *   other arguments as in rq_add_rmsnorm_nvfp4; no output may overlap an
 *   input.
 */
rq_status rq_gated_rmsnorm_nvfp4(const void *x, const void *z,
                                 const void *weight, float eps,
                                 const float *d_global_scale,
                                 uint8_t *q_packed, uint8_t *block_scales,
                                 void *norm_out, int64_t rows, int64_t hidden,
                                 rq_dtype dt, rq_stream_t stream);
/* The same with the block scales in the swizzled layout of
 * rq_add_rmsnorm_nvfp4_swizzled (rq_nvfp4_swizzled_scale_bytes bytes, every
 * byte written, padding 0). */
rq_status rq_gated_rmsnorm_nvfp4_swizzled(const void *x, const void *z,
                                          const void *weight, float eps,
                                          const float *d_global_scale,
                                          uint8_t *q_packed,
                                          uint8_t *block_scales, void *norm_out,
                                          int64_t rows, int64_t hidden,
                                          rq_dtype dt, rq_stream_t stream);

/*
 * Calibration: d_amax = max over the tensor of |y| (the norm output the
 * fused calls would produce), written to one device fp32.  Nothing else is
 * written.  The call clears d_amax on `stream` first (so an empty tensor
 * gives 0; x, residual_in and weight may then be NULL).
 * Source: the per-tensor scales the pages use are derived from the norm
 * output's absolute maximum ("Add AutoDeploy NVFP4 RMSNorm quant fusion",
 * Changes: reference module with input-scale calibration).
 */
rq_status rq_add_rmsnorm_amax(const void *x, const void *residual_in,
                              const void *weight, float eps, float *d_amax,
                              int64_t rows, int64_t hidden, rq_dtype dt,
                              rq_stream_t stream);

/* d_scale = amax / 448 (the FP8 dequant scale) and d_gs = 448 * 6 / amax
 * (the NVFP4 global scale), each one fp32 division on the device (the plain
 * formulas: a zero amax gives 0 and inf). */
rq_status rq_fp8_scale_from_amax(const float *d_amax, float *d_scale,
                                 rq_stream_t stream);
rq_status rq_nvfp4_global_scale_from_amax(const float *d_amax, float *d_gs,
                                          rq_stream_t stream);

/*
 * Dynamic scales (residual add + RMSNorm, then the quantiser with a scale
 * taken from the norm output itself).
 * Source: the pages' per-tensor scales are absolute maxima of the tensor
 * ("Add AutoDeploy NVFP4 RMSNorm quant fusion", Changes: reference module
 * with input-scale calibration); "Add NanoJet backend for AutoDeploy
 * prefill-only FP8 inference", Description: FP8 quantisation in the norm
 * epilogue.  A maximum of zero (all-zero row or tensor) gives the scale 1,
 * so that the codes are zeros rather than the 0/0 of the plain formula.
 *
 * rq_add_rmsnorm_fp8_per_token: one pass; row r gets the dequant scale
 *   d_row_scales[r] = amax_r(|y|) / 448 (fp32, written) and
 *   q = E4M3(y / d_row_scales[r]).  d_row_scales: [rows] fp32.
 * rq_add_rmsnorm_fp8_dynamic / rq_add_rmsnorm_nvfp4_dynamic: two passes over
 *   x and residual (the first finds the tensor's amax, the second is the
 *   fused call); *d_scale_out receives the scale used (FP8: amax / 448;
 *   NVFP4: 2688 / amax).  The first pass accumulates the maximum in
 *   *d_scale_out itself, so no workspace is needed.  In-place residual is
 *   allowed (the first pass only reads).
 * Other arguments as in rq_add_rmsnorm_fp8 / rq_add_rmsnorm_nvfp4.
 */
rq_status rq_add_rmsnorm_fp8_per_token(const void *x, const void *residual_in,
                                       void *residual_out, const void *weight,
                                       float eps, uint8_t *q_out,
                                       float *d_row_scales, void *norm_out,
                                       int64_t rows, int64_t hidden,
                                       rq_dtype dt, rq_stream_t stream);
rq_status rq_add_rmsnorm_fp8_dynamic(const void *x, const void *residual_in,
                                     void *residual_out, const void *weight,
                                     float eps, float *d_scale_out,
                                     uint8_t *q_out, void *norm_out,
                                     int64_t rows, int64_t hidden, rq_dtype dt,
                                     rq_stream_t stream);
rq_status rq_add_rmsnorm_nvfp4_dynamic(const void *x, const void *residual_in,
                                       void *residual_out, const void *weight,
                                       float eps, float *d_global_scale_out,
                                       uint8_t *q_packed, uint8_t *block_scales,
                                       void *norm_out, int64_t rows,
                                       int64_t hidden, rq_dtype dt,
                                       rq_stream_t stream);

/*
 * The NVFP4 calls with the block scales written in the layout a block-scaled
 * NVFP4 GEMM reads for an operand (cuBLASLt's 16-element-block / E4M3-scale
 * mode), so that no reordering pass runs between this call and the GEMM:
 *   - the rows x (hidden/16) matrix of block scales is padded to a multiple
 *     of 128 rows and of 4 block columns;
 *   - it is cut into 128 x 4 tiles of 512 bytes each, stored one row of
 *     tiles after the other, left to right within a row of tiles;
 *   - inside a tile, the scale of (row r, block column c) is byte
 *     16 * (r % 32) + 4 * (r / 32) + c.
 * Every byte of block_scales is written; the padding bytes are 0.
 *   block_scales  rq_nvfp4_swizzled_scale_bytes(rows, hidden) bytes
 * All other arguments, the outputs and the checks are those of
 * rq_add_rmsnorm_nvfp4 / rq_add_rmsnorm_nvfp4_dynamic; with rows == 0
 * nothing is written (the padded size is 0 too).
 * Source: the pages size the scale tensor for its GEMM ("Add AutoDeploy NVFP4
 * RMSNorm quant fusion", review: the sf_size math of the shape-only ops;
 * "[Performance]: Fuse local NVFP4 tail after NCCL fallback", Correctness
 * and build validation: the expected packed NVFP4 output shape) but do not
 * print the layout; it is the consumer's.
 */
rq_status rq_add_rmsnorm_nvfp4_swizzled(const void *x, const void *residual_in,
                                        void *residual_out, const void *weight,
                                        float eps, const float *d_global_scale,
                                        uint8_t *q_packed,
                                        uint8_t *block_scales, void *norm_out,
                                        int64_t rows, int64_t hidden,
                                        rq_dtype dt, rq_stream_t stream);
rq_status rq_add_rmsnorm_nvfp4_dynamic_swizzled(
    const void *x, const void *residual_in, void *residual_out,
    const void *weight, float eps, float *d_global_scale_out,
    uint8_t *q_packed, uint8_t *block_scales, void *norm_out, int64_t rows,
    int64_t hidden, rq_dtype dt, rq_stream_t stream);

/* Output sizes of the NVFP4 call (the linear, unswizzled layout):
 * rows * hidden / 2 packed bytes and rows * hidden / 16 scale bytes.
 * Source: "Add AutoDeploy NVFP4 RMSNorm quant fusion", review: the packed
 * output and scale-tensor size math of the fake (shape-only) ops. */
size_t rq_nvfp4_packed_bytes(int64_t rows, int64_t hidden);
size_t rq_nvfp4_scale_bytes(int64_t rows, int64_t hidden);
/* Block-scale bytes of the swizzled calls:
 * ceil(rows / 128) * 128 * ceil(hidden / 64) * 4. */
size_t rq_nvfp4_swizzled_scale_bytes(int64_t rows, int64_t hidden);

/* Text of a status code (static storage). */
const char *rq_status_string(rq_status status);

/* Message of the last RQ_ERR_CUDA returned on the calling thread (static,
 * thread-local storage; "" if none). */
const char *rq_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int rq_version(void);

#ifdef __cplusplus
}
#endif
#endif /* RQ_H */
