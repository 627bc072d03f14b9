/*
 * rq_oracle.h -- plain CPU oracle for the fused residual-add + RMSNorm +
 * FP8 / NVFP4 quantisation path and the per-head Q/K RMSNorm + RoPE + FP8
 * store.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a slow, single-threaded, obviously
 * correct restatement of what the path computes.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg load it.  The CUDA library shares
 * no code, header, table or helper with it, and never calls it.
 *
 * Sources (pages, by title and section):
 *   [P1] "Add NanoJet backend for AutoDeploy prefill-only FP8 inference"
 *        (TensorRT-LLM PR 17288), Description: RMSNorm with FP8 quantisation
 *        in the epilogue; fused Q/K RMSNorm and RoPE.
 *   [P2] "Add AutoDeploy NVFP4 RMSNorm quant fusion" (TensorRT-LLM PR 14361),
 *        Walkthrough / Changes: fused add + RMSNorm + NVFP4 ops, with and
 *        without the high-precision norm output.
 *   [P3] "perf: add fused norm + RoPE + uniform fp8 store for TRT-LLM DSv4
 *        sparse attention" (SGLang PR 32975), review thread: norm + RoPE +
 *        uniform FP8 store.
 *   [P4] "[Performance]: Fuse local NVFP4 tail after NCCL fallback"
 *        (TensorRT-LLM issue 17900), Proposal: residual + RMSNorm (+ norm
 *        output) + NVFP4 in one pass; support conditions (FP16/BF16, FP32
 *        per-tensor scale, hidden % 16 == 0).
 * The pages give the operations but not their rounding points; the readings
 * taken here (quantise from the dtype-rounded norm output, eps inside the
 * square root, plain multiply by the weight, IEEE division by the FP8 scale,
 * NVFP4 block scale = E4M3(gs*amax/6), encode factor gs/scale) are the plain
 * ones and are listed in the design notes.
 *
 * Storage types: bfloat16 / float16 are passed as uint16_t bit patterns,
 * E4M3 and packed E2M1 as uint8_t.  Every fp32 step is a C `float`
 * operation compiled with -ffp-contract=off, i.e. one IEEE single rounding
 * (round to nearest even) per operation.
 */
#ifndef RQ_ORACLE_H
#define RQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { RQO_BF16 = 0, RQO_FP16 = 1 };

/* ---- number formats (exact decoders, round-to-nearest-even encoders) ---- */
double   oracle_bf16_to_double(uint16_t b);
double   oracle_fp16_to_double(uint16_t h);
uint16_t oracle_bf16_from_double(double v);   /* RNE, overflow to +-inf */
uint16_t oracle_fp16_from_double(double v);   /* RNE, overflow to +-inf */
double   oracle_e4m3_to_double(uint8_t c);    /* OCP E4M3 (fn): bias 7, max 448 */
uint8_t  oracle_e4m3_from_double(double v);   /* RNE, satfinite to +-448 */
double   oracle_e2m1_to_double(uint8_t nib);  /* low 4 bits: sign<<3 | index */
uint8_t  oracle_e2m1_from_double(double v);   /* RNE, satfinite to +-6 */

/* Array forms of the encoders/decoders (used by the format tests). */
void oracle_dt_from_double_array(int dt, const double *v, int64_t n, uint16_t *out);
void oracle_dt_to_double_array(int dt, const uint16_t *b, int64_t n, double *out);
void oracle_e4m3_from_double_array(const double *v, int64_t n, uint8_t *out);
void oracle_e2m1_from_double_array(const double *v, int64_t n, uint8_t *out);

/* ---- residual add + RMSNorm ---------------------------------------------
 * Per row of `hidden` elements:
 *   s_i  = dt(f32(x_i) + f32(r_i))                       -> s_out (residual')
 *   ss   = f32(sum_i s_i^2)   (sum taken in double, rounded once)
 *   rstd = f32(1 / f32(sqrt(f32(f32(ss / hidden) + eps))))
 *   y_i  = dt(f32(f32(s_i * rstd) * w_i))                -> y_out (norm out)
 * s_out may equal r (in place).  y_out may be NULL. */
void oracle_add_rmsnorm(int dt, const uint16_t *x, const uint16_t *r,
                        const uint16_t *w, float eps, int64_t rows,
                        int64_t hidden, uint16_t *s_out, uint16_t *y_out);

/* Per-tensor FP8: q_i = E4M3sat(f32(y_i / scale)); scale is the dequant
 * scale (x ~= e4m3(q) * scale). */
void oracle_quant_fp8(int dt, const uint16_t *y, int64_t n, float scale,
                      uint8_t *q);

/* NVFP4 over rows of `hidden` (hidden % 16 == 0); gs = global scale in the
 * quantising direction (e.g. 448*6/amax).  Per 16-element block:
 *   a   = max_i |y_i|
 *   sf  = E4M3sat(f32(f32(gs * a) / 6))                  -> sf[row*hidden/16+b]
 *   enc = (sf == 0) ? 0 : f32(gs / sf)
 *   c_i = E2M1sat(f32(y_i * enc)),  byte j = c_2j | c_2j+1 << 4 -> packed
 * Dequantised value: e2m1(c_i) * sf / gs. */
void oracle_quant_nvfp4(int dt, const uint16_t *y, int64_t rows,
                        int64_t hidden, float gs, uint8_t *packed,
                        uint8_t *sf);

/* Whole fused calls: residual add + RMSNorm, then the quantiser. */
void oracle_add_rmsnorm_fp8(int dt, const uint16_t *x, const uint16_t *r,
                            const uint16_t *w, float eps, float scale,
                            int64_t rows, int64_t hidden, uint16_t *s_out,
                            uint16_t *y_out, uint8_t *q);
void oracle_add_rmsnorm_nvfp4(int dt, const uint16_t *x, const uint16_t *r,
                              const uint16_t *w, float eps, float gs,
                              int64_t rows, int64_t hidden, uint16_t *s_out,
                              uint16_t *y_out, uint8_t *packed, uint8_t *sf);

/* Gated RMSNorm + NVFP4 ([P2] Changes: the fused gated RMSNorm + NVFP4 op;
 * its formula is not on the page).  Reading: the separated sequence the
 * fused op replaces, gate applied before the norm, one norm group per row,
 * no residual:
 *   silu(z) = z / (1 + e^-z), rounded to fp32 and then to the dtype
 *   g_i     = dt(f32(x_i * silu(z_i)))                  -> g_out
 *   then the RMSNorm steps above with residual' := g    -> y_out
 *   and oracle_quant_nvfp4 on y (the _nvfp4 variant). */
uint16_t oracle_silu_dt(int dt, uint16_t z);
void oracle_gated_rmsnorm(int dt, const uint16_t *x, const uint16_t *z,
                          const uint16_t *w, float eps, int64_t rows,
                          int64_t hidden, uint16_t *g_out, uint16_t *y_out);
void oracle_gated_rmsnorm_nvfp4(int dt, const uint16_t *x, const uint16_t *z,
                                const uint16_t *w, float eps, float gs,
                                int64_t rows, int64_t hidden, uint16_t *g_out,
                                uint16_t *y_out, uint8_t *packed, uint8_t *sf);

/* GEMM-facing block-scale layout.  The pages size the block-scale tensor for
 * the GEMM that consumes it ("Add AutoDeploy NVFP4 RMSNorm quant fusion",
 * review: the sf_size math of the shape-only ops; "[Performance]: Fuse local
 * NVFP4 tail after NCCL fallback", Correctness: the expected packed NVFP4
 * output shape) but do not print the layout.  The one written here is the
 * layout the block-scaled NVFP4 GEMM of cuBLASLt (16-element blocks, E4M3
 * scales) reads for an operand: the rows x nb scale matrix (nb = hidden/16)
 * is padded with zero bytes to a multiple of 128 rows and of 4 block
 * columns and cut into 128 x 4 tiles of 512 bytes, stored with the row of
 * tiles outermost; inside a tile the scale of (row r, block column c) is
 * byte 16*(r mod 32) + 4*(r div 32) + c.  Pinned by feeding its output to
 * that GEMM (GPU test), not by the pages.
 *   sf:  [rows, hidden/16] linear scales (as oracle_quant_nvfp4 writes them)
 *   out: oracle_nvfp4_swizzled_scale_bytes(rows, hidden) bytes, all written */
int64_t oracle_nvfp4_swizzled_scale_bytes(int64_t rows, int64_t hidden);
void oracle_nvfp4_swizzle_scales(const uint8_t *sf, int64_t rows,
                                 int64_t hidden, uint8_t *out);

/* Dynamic scales.  A scale derived from an absolute maximum of zero (an
 * all-zero row or tensor) is taken as 1, so that every code is a signed zero
 * and the dequantised values are zero, instead of the 0/0 of the plain
 * formula.
 *   per row:    scale_r = f32(amax_r / 448), q = E4M3sat(f32(y / scale_r))
 *   per tensor: scale = f32(amax / 448) (FP8), gs = f32(2688 / amax) (NVFP4) */
void oracle_quant_fp8_per_row(int dt, const uint16_t *y, int64_t rows,
                              int64_t hidden, uint8_t *q, float *row_scales);
float oracle_fp8_dynamic_scale(float amax);
float oracle_nvfp4_dynamic_gs(float amax);

/* max_i |v_i| of a dtype tensor (exact), and the calibrated scales. */
float oracle_amax(int dt, const uint16_t *v, int64_t n);
float oracle_fp8_scale_from_amax(float amax);    /* f32(amax / 448)  */
float oracle_nvfp4_gs_from_amax(float amax);     /* f32(2688 / amax) */

/* ---- per-head Q/K RMSNorm + NeoX RoPE (+ FP8) -----------------------------
 * src: n_tokens tokens, token t starts at src + t*token_stride elements and
 * holds n_heads contiguous heads of head_dim elements.  For each head:
 *   n   = RMSNorm of the head (same steps as above, weight w[head_dim],
 *         no residual), rounded to dt
 *   p   = clamp(pos[t], 0, max_pos-1); c_i = cs[p][i], s_i = cs[p][half+i]
 *   o_i        = dt(f32(f32(n_i * c_i) - f32(n_{i+half} * s_i)))
 *   o_{i+half} = dt(f32(f32(n_{i+half} * c_i) + f32(n_i * s_i)))
 * with half = head_dim/2 and cs a [max_pos, head_dim] fp32 table
 * (cos in the first half, sin in the second).  o is written densely as
 * [n_tokens, n_heads, head_dim]. */
void oracle_qk_rmsnorm_rope(int dt, const uint16_t *src, int64_t token_stride,
                            int64_t n_tokens, int n_heads, int head_dim,
                            const uint16_t *w, float eps, const int32_t *pos,
                            const float *cos_sin, int64_t max_pos,
                            uint16_t *o);
/* The above followed by oracle_quant_fp8 with `scale`. */
void oracle_qk_rmsnorm_rope_fp8(int dt, const uint16_t *src,
                                int64_t token_stride, int64_t n_tokens,
                                int n_heads, int head_dim, const uint16_t *w,
                                float eps, const int32_t *pos,
                                const float *cos_sin, int64_t max_pos,
                                float scale, uint16_t *o, uint8_t *q);

/* ---- Q/K RMSNorm + NeoX RoPE over part of the head --------------------------
 * The FP8-nope + BF16-rope KV pool that "perf: add fused norm + RoPE + uniform
 * fp8 store for TRT-LLM DSv4 sparse attention" (SGLang PR 32975, review
 * thread) names for the FlashMLA path.  The page does not give the split of a
 * head; the reading taken: each head is [nope | rope] with the rotated part
 * the LAST rope_dim elements.  Per head:
 *   n   = RMSNorm of the whole head (as above), rounded to dt
 *   o_i = n_i                                          for i < nope
 *   with j = nope + i, i < rope_dim/2, c = cs[p][i], s = cs[p][rope_dim/2 + i]:
 *   o_j              = dt(f32(f32(n_j * c) - f32(n_{j+rope_dim/2} * s)))
 *   o_{j+rope_dim/2} = dt(f32(f32(n_{j+rope_dim/2} * c) + f32(n_j * s)))
 * with nope = head_dim - rope_dim and cs a [max_pos, rope_dim] fp32 table
 * (rope_dim/2 cos, then rope_dim/2 sin).  rope_dim == head_dim is the call
 * above.  In the KV pool the nope part is stored as E4M3 (oracle_quant_fp8)
 * and the rope part as the dtype values o. */
void oracle_qk_rmsnorm_rope_partial(int dt, const uint16_t *src,
                                    int64_t token_stride, int64_t n_tokens,
                                    int n_heads, int head_dim, int rope_dim,
                                    const uint16_t *w, float eps,
                                    const int32_t *pos, const float *cos_sin,
                                    int64_t max_pos, uint16_t *o);

#ifdef __cplusplus
}
#endif
#endif /* RQ_ORACLE_H */
