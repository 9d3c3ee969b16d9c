/*
 * mxfp4_oracle.h — plain, slow, single-threaded CPU oracle of MXFP4 block
 * quantization.  TEST INFRASTRUCTURE ONLY: it exists so that tests, the
 * smoke check and the CPU-baseline leg of the benchmark can check the GPU
 * library against an obviously correct restatement of the method.  The
 * product library never links, loads or calls it, and it shares no source
 * with the GPU path.
 *
 * Every function names the passage it follows:
 *   [PR43557] vLLM PR #43557 page, "Fix the E8M0 scale computation in the
 *             MXFP4 MoE CUTLASS kernel" (sections named per function).
 *   [PR51038] vLLM PR #51038 page, "[Bugfix][Quantization] Fix MXFP4
 *             conversion for FlashInfer CUTLASS".
 *   [PR46915] vLLM PR #46915 page, "Fix the SM90 MXFP4 MoE test weight/scale
 *             interleave".
 * Steps the pages leave open follow the OCP MX v1.0 definition of E2M1 and
 * E8M0, as noted per function.
 *
 * Parity pins: every function here is checked by the CPU test-suite against
 * something other than itself (closed forms, exhaustive enumeration against an
 * independent formulation, the pages' own worked tensors).  The reporting
 * helpers (relative L2 error, saturation count) are computed by the tests
 * from oracle outputs and carry no pin of their own: parity unpinned.
 */
#ifndef MXFP4_ORACLE_H
#define MXFP4_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* BF16 bit pattern -> exact double. */
double orc_bf16_to_double(uint16_t b);
/* double -> BF16 bit pattern, round to nearest, ties to even; overflow to
 * +-Inf, subnormals kept, NaN -> 0x7FC0 (sign kept). */
uint16_t orc_double_to_bf16_rne(double d);

/* Step 1: vecMax = max |x| over n BF16 values, as a float (exact). */
float orc_block_absmax(const uint16_t* x, int64_t n);
/* Step 2: E8M0 scale exponent of a block from its vecMax. */
uint8_t orc_e8m0_scale(float vecmax);
/* Steps 3: E2M1 nibble of one BF16 element under scale exponent s. */
uint8_t orc_e2m1_encode(uint16_t xbits, uint8_t s);
/* FP16 input: exact value of a binary16 pattern; nibble of one element. */
double orc_f16_to_double(uint16_t h);
uint8_t orc_e2m1_encode_f16(uint16_t hbits, uint8_t s);
/* E2M1 nibble -> exact value (sign kept, code 0x8 is -0.0). */
double orc_e2m1_decode(uint8_t nib);

/* Vector forms used by the exhaustive pins. */
void orc_e8m0_scale_many(const uint16_t* vbits, int64_t n, uint8_t* s);
void orc_e2m1_encode_many(const uint16_t* x, int64_t n, uint8_t s, uint8_t* nib);
void orc_dequant_value_many(const uint8_t* nib, const uint8_t* s, int64_t n, uint16_t* y);
void orc_e2m1_encode_f16_many(const uint16_t* x, int64_t n, uint8_t s, uint8_t* nib);
void orc_f16_to_double_many(const uint16_t* x, int64_t n, double* out);

/* Tiled scale size: ceil(M/128)*128 * ceil(sK/4)*4 bytes, sK = K/32. */
size_t orc_scale_bytes(int64_t M, int64_t K);

/* Steps 1-4: flat per-block scales [M, K/32] and packed codes [M, K/2]. */
void orc_quantize_flat(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                       uint8_t* codes, uint8_t* flat_scales);
/* Comparison only: the pre-fix scale biased_exp(vecMax/6) and steps 1-4 with it. */
uint8_t orc_e8m0_scale_legacy(float vecmax);
void orc_quantize_flat_legacy(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                              uint8_t* codes, uint8_t* flat_scales);
/* Step 5: flat [M, sK] scales <-> CUTLASS 128x4 tiled, zero-padded bytes. */
void orc_tile_scales(const uint8_t* flat, int64_t M, int64_t sK, uint8_t* tiled);
void orc_untile_scales(const uint8_t* tiled, int64_t M, int64_t sK, uint8_t* flat);
/* Steps 1-5 together: codes + tiled scales (orc_scale_bytes(M,K) bytes). */
void orc_quantize(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                  uint8_t* codes, uint8_t* tiled_scales);
/* Steps 1-5 for FP16 input [M, K] (row stride ldx). */
void orc_quantize_flat_f16(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                           uint8_t* codes, uint8_t* flat_scales);
void orc_quantize_f16(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                      uint8_t* codes, uint8_t* tiled_scales);
/* Step 6: per-segment quantize.  Returns 0, or -6 when the offsets break
 * 0 = o[0] <= ... <= o[E] = total_rows (then scale_row_offsets = -1 and
 * codes/scales are untouched). */
int orc_quantize_grouped(const uint16_t* x, int64_t total_rows, int64_t K,
                         const int32_t* offsets, int32_t E, uint8_t* codes,
                         uint8_t* scales, int32_t* scale_row_offsets);
/* Step 6 on gathered rows: output row r is row row_index[r] of x (row
 * stride ldx).  Returns 0, -6 (bad offsets, as above) or -7 (some index
 * outside [0, num_src_rows): that row is quantized as zeros). */
int orc_quantize_grouped_gather(const uint16_t* x, int64_t num_src_rows, int64_t K, int64_t ldx,
                                const int32_t* row_index, int64_t total_rows,
                                const int32_t* offsets, int32_t E, uint8_t* codes,
                                uint8_t* scales, int32_t* scale_row_offsets);
int orc_quantize_grouped_scatter(const uint16_t* x, int64_t num_tokens, int64_t K, int64_t ldx,
                                 const int32_t* dest_rows, int32_t top_k, int64_t total_rows,
                                 const int32_t* offsets, int32_t E, uint8_t* codes,
                                 uint8_t* scales, int32_t* scale_row_offsets);
/* FP16 input for the three grouped forms (segments quantized as orc_quantize_f16). */
int orc_quantize_grouped_f16(const uint16_t* x, int64_t total_rows, int64_t K,
                             const int32_t* offsets, int32_t E, uint8_t* codes,
                             uint8_t* scales, int32_t* scale_row_offsets);
int orc_quantize_grouped_gather_f16(const uint16_t* x, int64_t num_src_rows, int64_t K,
                                    int64_t ldx, const int32_t* row_index, int64_t total_rows,
                                    const int32_t* offsets, int32_t E, uint8_t* codes,
                                    uint8_t* scales, int32_t* scale_row_offsets);
int orc_quantize_grouped_scatter_f16(const uint16_t* x, int64_t num_tokens, int64_t K,
                                     int64_t ldx, const int32_t* dest_rows, int32_t top_k,
                                     int64_t total_rows, const int32_t* offsets, int32_t E,
                                     uint8_t* codes, uint8_t* scales,
                                     int32_t* scale_row_offsets);
/* Step 7: codes + tiled scales -> BF16 [M, K]. */
void orc_dequantize(const uint8_t* codes, const uint8_t* tiled_scales,
                    int64_t M, int64_t K, uint16_t* y);
/* Step 8 parts: swap the two row halves of each of E [two_n, row_bytes]
 * byte matrices; swap the halves of each [two_n] bias row and cast it to BF16;
 * cast a plain FP32 vector to BF16 (RNE). */
void orc_swap_halves(const uint8_t* in, uint8_t* out, int64_t E, int64_t two_n,
                     int64_t row_bytes);
void orc_swap_bias_bf16(const float* in, uint16_t* out, int64_t E, int64_t two_n);
void orc_cast_bf16(const float* in, uint16_t* out, int64_t n);
/* Step 8: [w1; w3] -> [w3; w1] for codes, scales and biases. */
void orc_swap_w13(const uint8_t* codes_in, const uint8_t* scales_in,
                  const float* w13_bias_in, int32_t E, int64_t two_n, int64_t K,
                  int32_t scales_tiled, uint8_t* codes_out, uint8_t* scales_out,
                  uint16_t* w13_bias_out, const float* w2_bias_in,
                  int64_t w2_bias_numel, uint16_t* w2_bias_out);

/* NVFP4 (16-element blocks, E4M3 block scale, caller's global scale g). */
double orc_e4m3_to_double(uint8_t b);
uint8_t orc_e4m3_from_double(double d);
void orc_e4m3_from_double_many(const double* d, int64_t n, uint8_t* out);
size_t orc_nvfp4_scale_bytes(int64_t M, int64_t K);
void orc_nvfp4_quantize_flat(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, float g,
                             uint8_t* codes, uint8_t* flat_scales);
void orc_nvfp4_quantize(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, float g,
                        uint8_t* codes, uint8_t* tiled_scales);
/* NVFP4 experts quant: per-segment NVFP4 with per-segment global scales g[E]
 * in the grouped scale layout; returns 0 or -6 (bad offsets). */
int orc_nvfp4_quantize_grouped(const uint16_t* x, int64_t total_rows, int64_t K,
                               const int32_t* offsets, int32_t E, const float* g,
                               uint8_t* codes, uint8_t* scales, int32_t* scale_row_offsets);
/* NVFP4 on IEEE binary16 input (dense and experts quant). */
void orc_nvfp4_quantize_f16(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, float g,
                            uint8_t* codes, uint8_t* tiled_scales);
int orc_nvfp4_quantize_grouped_f16(const uint16_t* x, int64_t total_rows, int64_t K,
                                   const int32_t* offsets, int32_t E, const float* g,
                                   uint8_t* codes, uint8_t* scales, int32_t* scale_row_offsets);
/* NVFP4 experts quant with the dispatch as a scatter (route j of token t ->
 * row dest_rows[t * top_k + j], -1 = none): untargeted rows keep their bytes,
 * pad rows zero scales; returns 0, -6 (bad offsets) or -7 (bad entries). */
int orc_nvfp4_quantize_grouped_scatter(const uint16_t* x, int64_t num_tokens, int64_t K,
                                       int64_t ldx, const int32_t* dest_rows, int32_t top_k,
                                       int64_t total_rows, const int32_t* offsets, int32_t E,
                                       const float* g, uint8_t* codes, uint8_t* scales,
                                       int32_t* scale_row_offsets);
int orc_nvfp4_quantize_grouped_scatter_f16(const uint16_t* x, int64_t num_tokens, int64_t K,
                                           int64_t ldx, const int32_t* dest_rows, int32_t top_k,
                                           int64_t total_rows, const int32_t* offsets, int32_t E,
                                           const float* g, uint8_t* codes, uint8_t* scales,
                                           int32_t* scale_row_offsets);
void orc_nvfp4_dequantize(const uint8_t* codes, const uint8_t* tiled_scales, int64_t M, int64_t K,
                          float g, uint16_t* y);
/* The dispatch permutation from the router's expert ids [num_tokens, top_k]:
 * rows in order of expert, then of entry index; offsets [E+1], dest_rows
 * [num_tokens * top_k] (-1: not dispatched), row_index [rows] (may be NULL).
 * Returns 0 or -7 (an id neither -1 nor in [0, E); it is not dispatched). */
int orc_moe_route(const int32_t* topk_ids, int64_t num_tokens, int32_t top_k, int32_t E,
                  int32_t* offsets, int32_t* dest_rows, int32_t* row_index);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_ORACLE_H */
