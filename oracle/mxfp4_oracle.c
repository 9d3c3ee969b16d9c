/*
 * mxfp4_oracle.c — plain single-threaded CPU oracle of MXFP4 block
 * quantization.  TEST INFRASTRUCTURE ONLY (tests, smoke check, the CPU
 * baseline of the benchmark); the GPU library never uses it.  Written for a
 * reader checking it against the pages by eye: no blocking, no fusion, one
 * step per function, doubles wherever the value is exact.
 *
 * Sources: see mxfp4_oracle.h ([PR43557], [PR51038], [PR46915]).
 */
#include "mxfp4_oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* float expressions must round every operation to float (x86-64 SSE, AArch64) */
_Static_assert(FLT_EVAL_METHOD == 0, "float arithmetic must be evaluated in float");

/* ---------------------------------------------------------------------- */
/* BF16 helpers (IEEE binary32 with the low 16 mantissa bits dropped).     */

double orc_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

uint16_t orc_double_to_bf16_rne(double d) {
  uint16_t sign = signbit(d) ? 0x8000u : 0u;
  double a = fabs(d);
  if (isnan(d)) return (uint16_t)(sign | 0x7FC0u);
  if (a == 0.0) return sign;
  if (isinf(d)) return (uint16_t)(sign | 0x7F80u);
  /* Quantum (spacing of BF16 values) around a: 2^-133 in the subnormal
   * range, else 2^(e-7) with e = floor(log2 a). */
  int e;
  frexp(a, &e); /* a = f * 2^e, f in [0.5, 1)  ->  floor(log2 a) = e - 1 */
  int exp2 = e - 1;
  int qexp = (exp2 < -126) ? -133 : exp2 - 7;
  double n = nearbyint(ldexp(a, -qexp)); /* ties to even (default mode) */
  double r = ldexp(n, qexp);
  if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);
  if (r < ldexp(1.0, -126)) return (uint16_t)(sign | (uint16_t)n); /* subnormal */
  frexp(r, &e);
  int rexp = e - 1;                                  /* r in [2^rexp, 2^(rexp+1)) */
  uint32_t mant = (uint32_t)(ldexp(r, -rexp) * 128.0 - 128.0);
  return (uint16_t)(sign | ((uint32_t)(rexp + 127) << 7) | mant);
}

static float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* ---------------------------------------------------------------------- */
/* Step 1 — block absmax.  [PR43557] cvt_warp_fp16_to_fp4 excerpt: vecMax is
 * the block's largest magnitude, taken as a float.  |x| clears the sign bit;
 * a max involves no rounding. */
float orc_block_absmax(const uint16_t* x, int64_t n) {
  float v = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float a = bf16_to_float((uint16_t)(x[i] & 0x7FFFu));
    if (a > v) v = a;
  }
  return v;
}

/* Step 2 — E8M0 scale.  [PR43557] "Implementation breakdown" item 1 and the
 * UE8M0 branch of the cvt_warp_fp16_to_fp4 excerpt (also its Python form,
 * compute_reference_e8m0_scale): round the mantissa of vecMax up when it is
 * >= 0.75 by adding 2^21 to its IEEE-754 bits, keep the sign+exponent field,
 * take the biased exponent, subtract 2 (never below 0), cap at 254.  A block
 * whose max is <= 0 gets 0. */
uint8_t orc_e8m0_scale(float vecmax) {
  if (vecmax <= 0.0f) return 0;
  uint32_t bits;
  memcpy(&bits, &vecmax, sizeof bits);
  uint32_t rounded = (bits + (1u << 21)) & 0xFF800000u; /* 32-bit wraparound */
  uint32_t biased_exp = (rounded >> 23) & 0xFFu;
  uint32_t s = (biased_exp > 2u) ? biased_exp - 2u : 0u;
  if (s > 254u) s = 254u;
  return (uint8_t)s;
}

/* Step 3 — one element.  The pages fix only the E2M1 range (largest
 * magnitude 6.0, [PR43557] "Motivation") and the scale value 2^(s-127)
 * (the SFValue line of the excerpt).  Plain OCP-MX reading: divide by the
 * scale (an exact power of two), round the magnitude to the nearest of
 * {0, 0.5, 1, 1.5, 2, 3, 4, 6}, ties to the value with an even mantissa bit
 * (the even index), anything above 6 stays 6 (saturation); keep the sign
 * (so -0.0 and small negatives give 0x8).  Blocks with s == 0 emit 0x0 for
 * every element (the convention fixed for this library). */
static uint8_t e2m1_round(double y, int negative) {
  double m = fabs(y);
  uint8_t idx;
  /* midpoints 0.25 0.75 1.25 1.75 2.5 3.5 5; at a tie the even index wins */
  if (m <= 0.25) idx = 0;        /* 0.25 ties 0 (idx 0) / 0.5 (idx 1)   */
  else if (m < 0.75) idx = 1;    /* 0.75 ties 0.5 (1) / 1.0 (2)         */
  else if (m <= 1.25) idx = 2;   /* 1.25 ties 1.0 (2) / 1.5 (3)         */
  else if (m < 1.75) idx = 3;    /* 1.75 ties 1.5 (3) / 2.0 (4)         */
  else if (m <= 2.5) idx = 4;    /* 2.5  ties 2.0 (4) / 3.0 (5)         */
  else if (m < 3.5) idx = 5;     /* 3.5  ties 3.0 (5) / 4.0 (6)         */
  else if (m <= 5.0) idx = 6;    /* 5.0  ties 4.0 (6) / 6.0 (7)         */
  else idx = 7;                  /* (5, inf): 6.0, saturating           */
  return (uint8_t)(((negative ? 1u : 0u) << 3) | idx);
}

static uint8_t e2m1_of_scaled(double x, int negative, uint8_t s) {
  if (s == 0) return 0;
  return e2m1_round(ldexp(x, 127 - (int)s), negative); /* x / 2^(s-127), exact */
}

uint8_t orc_e2m1_encode(uint16_t xbits, uint8_t s) {
  return e2m1_of_scaled(orc_bf16_to_double(xbits), (xbits >> 15) & 1u, s);
}

/* FP16 (IEEE binary16) input, the other 16-bit type the pages' kernel name
 * (cvt_warp_fp16_to_fp4) and its packed half2 max refer to ([PR43557]
 * excerpt).  Exact value of the bit pattern: sign, 5-bit exponent (bias 15),
 * 10-bit mantissa; exponent 0 is subnormal (mantissa * 2^-24). */
double orc_f16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int m = h & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp(1024.0 + m, e - 25);
  return sign ? -v : v;
}

uint8_t orc_e2m1_encode_f16(uint16_t hbits, uint8_t s) {
  return e2m1_of_scaled(orc_f16_to_double(hbits), (hbits >> 15) & 1u, s);
}

/* E2M1 decode (OCP MX): bit 3 sign, bits 2..1 exponent (bias 1), bit 0
 * mantissa; exponent 0 is subnormal (0.5 * mantissa). */
double orc_e2m1_decode(uint8_t nib) {
  int sign = (nib >> 3) & 1;
  int e = (nib >> 1) & 3;
  int m = nib & 1;
  double mag = (e == 0) ? 0.5 * m : (1.0 + 0.5 * m) * ldexp(1.0, e - 1);
  return sign ? -mag : mag;
}

void orc_e8m0_scale_many(const uint16_t* vbits, int64_t n, uint8_t* s) {
  for (int64_t i = 0; i < n; ++i) s[i] = orc_e8m0_scale(bf16_to_float(vbits[i]));
}

void orc_e2m1_encode_many(const uint16_t* x, int64_t n, uint8_t s, uint8_t* nib) {
  for (int64_t i = 0; i < n; ++i) nib[i] = orc_e2m1_encode(x[i], s);
}

void orc_e2m1_encode_f16_many(const uint16_t* x, int64_t n, uint8_t s, uint8_t* nib) {
  for (int64_t i = 0; i < n; ++i) nib[i] = orc_e2m1_encode_f16(x[i], s);
}

void orc_f16_to_double_many(const uint16_t* x, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_double(x[i]);
}

/* Step 7 for one element: E2M1 value times the E8M0 value 2^(s-127), rounded
 * once to BF16; s == 255 is the E8M0 NaN. */
static uint16_t dequant_value(uint8_t nib, uint8_t s) {
  if (s == 255) return 0x7FC0u;
  double v = orc_e2m1_decode(nib) * ldexp(1.0, (int)s - 127);
  return orc_double_to_bf16_rne(v);
}

void orc_dequant_value_many(const uint8_t* nib, const uint8_t* s, int64_t n, uint16_t* y) {
  for (int64_t i = 0; i < n; ++i) y[i] = dequant_value(nib[i], s[i]);
}

/* ---------------------------------------------------------------------- */
/* Matrices.                                                               */

size_t orc_scale_bytes(int64_t M, int64_t K) {
  if (M <= 0 || K <= 0 || K % 32 != 0) return 0;
  int64_t sK = K / 32;
  int64_t padded_M = (M + 127) / 128 * 128;
  int64_t padded_sK = (sK + 3) / 4 * 4;
  return (size_t)(padded_M * padded_sK);
}

/* Steps 1-4 row by row, block by block: absmax, scale, 32 nibbles, then two
 * nibbles per byte with element 2j in the low half. */
void orc_quantize_flat(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                       uint8_t* codes, uint8_t* flat_scales) {
  int64_t sK = K / 32;
  for (int64_t r = 0; r < M; ++r) {
    const uint16_t* row = x + r * ldx;
    for (int64_t b = 0; b < sK; ++b) {
      const uint16_t* blk = row + b * 32;
      uint8_t s = orc_e8m0_scale(orc_block_absmax(blk, 32));
      flat_scales[r * sK + b] = s;
      uint8_t nib[32];
      for (int i = 0; i < 32; ++i) nib[i] = orc_e2m1_encode(blk[i], s);
      for (int j = 0; j < 16; ++j)
        codes[r * (K / 2) + b * 16 + j] = (uint8_t)(nib[2 * j] | (nib[2 * j + 1] << 4));
    }
  }
}

/* The scale the fix replaced, reproduced for comparison only ([PR43557]
 * "Motivation": the old code took the biased exponent of max/6, and since
 * floor(log2(a/b)) differs from floor(log2 a) - floor(log2 b) that scale is
 * one too small for most inputs, leaving max/scale above 6).  Reading: the
 * exponent field of the float32 quotient vecMax/6 (rounded to nearest),
 * 0 for a zero block.  Never used by the library. */
uint8_t orc_e8m0_scale_legacy(float vecmax) {
  if (vecmax <= 0.0f) return 0;
  float q = vecmax / 6.0f;
  uint32_t bits;
  memcpy(&bits, &q, sizeof bits);
  return (uint8_t)((bits >> 23) & 0xFFu);
}

/* Steps 1-4 with the legacy scale in place of step 2 (comparison only). */
void orc_quantize_flat_legacy(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                              uint8_t* codes, uint8_t* flat_scales) {
  int64_t sK = K / 32;
  for (int64_t r = 0; r < M; ++r) {
    const uint16_t* row = x + r * ldx;
    for (int64_t b = 0; b < sK; ++b) {
      const uint16_t* blk = row + b * 32;
      uint8_t s = orc_e8m0_scale_legacy(orc_block_absmax(blk, 32));
      flat_scales[r * sK + b] = s;
      uint8_t nib[32];
      for (int i = 0; i < 32; ++i) nib[i] = orc_e2m1_encode(blk[i], s);
      for (int j = 0; j < 16; ++j)
        codes[r * (K / 2) + b * 16 + j] = (uint8_t)(nib[2 * j] | (nib[2 * j + 1] << 4));
    }
  }
}

/* Steps 1-4 for FP16 input: the same block max (as a float: every FP16
 * value is exact in float32), the same E8M0 rule on its float bits, the same
 * element rounding. */
void orc_quantize_flat_f16(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                           uint8_t* codes, uint8_t* flat_scales) {
  int64_t sK = K / 32;
  for (int64_t r = 0; r < M; ++r) {
    const uint16_t* row = x + r * ldx;
    for (int64_t b = 0; b < sK; ++b) {
      const uint16_t* blk = row + b * 32;
      float vmax = 0.0f;
      for (int i = 0; i < 32; ++i) {
        float a = (float)fabs(orc_f16_to_double(blk[i]));
        if (a > vmax) vmax = a;
      }
      uint8_t s = orc_e8m0_scale(vmax);
      flat_scales[r * sK + b] = s;
      uint8_t nib[32];
      for (int i = 0; i < 32; ++i) nib[i] = orc_e2m1_encode_f16(blk[i], s);
      for (int j = 0; j < 16; ++j)
        codes[r * (K / 2) + b * 16 + j] = (uint8_t)(nib[2 * j] | (nib[2 * j + 1] << 4));
    }
  }
}

/* Step 5 — CUTLASS 128x4 tiled scale layout.  [PR43557] untile_cutlass_scale:
 * the tiled bytes are viewed as [numMTiles, numKTiles, 32, 4, 4] and
 * permuted (0,3,2,1,4) back to [padded_M, padded_sK]; hence flat element
 * (r, c) lives at tiled index [r/128, c/4, r%32, (r%128)/32, c%4].  Bytes
 * outside [M, sK] but inside the padded extent are 0 (padding value: the
 * pages show the extent only; zero is this library's convention). */
static int64_t tiled_index(int64_t r, int64_t c, int64_t num_k_tiles) {
  int64_t m_tile = r / 128, k_tile = c / 4;
  int64_t outer_m = r % 32, inner_m = (r % 128) / 32, inner_k = c % 4;
  return (((m_tile * num_k_tiles + k_tile) * 32 + outer_m) * 4 + inner_m) * 4 + inner_k;
}

void orc_tile_scales(const uint8_t* flat, int64_t M, int64_t sK, uint8_t* tiled) {
  int64_t padded_M = (M + 127) / 128 * 128;
  int64_t num_k_tiles = (sK + 3) / 4;
  int64_t padded_sK = num_k_tiles * 4;
  for (int64_t r = 0; r < padded_M; ++r)
    for (int64_t c = 0; c < padded_sK; ++c)
      tiled[tiled_index(r, c, num_k_tiles)] = (r < M && c < sK) ? flat[r * sK + c] : 0;
}

void orc_untile_scales(const uint8_t* tiled, int64_t M, int64_t sK, uint8_t* flat) {
  int64_t num_k_tiles = (sK + 3) / 4;
  for (int64_t r = 0; r < M; ++r)
    for (int64_t c = 0; c < sK; ++c) flat[r * sK + c] = tiled[tiled_index(r, c, num_k_tiles)];
}

void orc_quantize(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                  uint8_t* codes, uint8_t* tiled_scales) {
  int64_t sK = K / 32;
  if (M <= 0 || sK <= 0) return;
  uint8_t* flat = (uint8_t*)calloc((size_t)(M * sK), 1);
  orc_quantize_flat(x, M, K, ldx, codes, flat);
  orc_tile_scales(flat, M, sK, tiled_scales);
  free(flat);
}

void orc_quantize_f16(const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                      uint8_t* codes, uint8_t* tiled_scales) {
  int64_t sK = K / 32;
  if (M <= 0 || sK <= 0) return;
  uint8_t* flat = (uint8_t*)calloc((size_t)(M * sK), 1);
  orc_quantize_flat_f16(x, M, K, ldx, codes, flat);
  orc_tile_scales(flat, M, sK, tiled_scales);
  free(flat);
}

/* Step 6 — per-expert ("experts quant") segments.  [PR43557] "Implementation
 * breakdown" item 3 tests the experts-quant kernel per block after untiling;
 * this library's reading: every segment [o[e], o[e+1]) is quantized as its
 * own matrix, codes keep the row order, and segment e's tiled scales (padded
 * to a multiple of 128 rows by itself) start at padded row P[e]. */
typedef void (*dense_quantize_fn)(const uint16_t*, int64_t, int64_t, int64_t, uint8_t*, uint8_t*);

static int grouped_with(dense_quantize_fn quantize, const uint16_t* x, int64_t total_rows,
                        int64_t K, const int32_t* offsets, int32_t E, uint8_t* codes,
                        uint8_t* scales, int32_t* scale_row_offsets) {
  int ok = (E >= 0) && offsets[0] == 0 && (int64_t)offsets[E] == total_rows;
  for (int32_t e = 0; ok && e < E; ++e) ok = offsets[e] <= offsets[e + 1];
  if (!ok) {
    for (int32_t e = 0; e <= E; ++e) scale_row_offsets[e] = -1;
    return -6;
  }
  int64_t sK = K / 32;
  int64_t padded_sK = (sK + 3) / 4 * 4;
  int64_t P = 0;
  for (int32_t e = 0; e < E; ++e) {
    int64_t n = (int64_t)offsets[e + 1] - offsets[e];
    scale_row_offsets[e] = (int32_t)P;
    quantize(x + (int64_t)offsets[e] * K, n, K, K, codes + (int64_t)offsets[e] * (K / 2),
             scales + P * padded_sK);
    P += (n + 127) / 128 * 128;
  }
  scale_row_offsets[E] = (int32_t)P;
  return 0;
}

int orc_quantize_grouped(const uint16_t* x, int64_t total_rows, int64_t K,
                         const int32_t* offsets, int32_t E, uint8_t* codes,
                         uint8_t* scales, int32_t* scale_row_offsets) {
  return grouped_with(orc_quantize, x, total_rows, K, offsets, E, codes, scales,
                      scale_row_offsets);
}

/* The same for FP16 input (segments quantized by the FP16 dense quantize). */
int orc_quantize_grouped_f16(const uint16_t* x, int64_t total_rows, int64_t K,
                             const int32_t* offsets, int32_t E, uint8_t* codes,
                             uint8_t* scales, int32_t* scale_row_offsets) {
  return grouped_with(orc_quantize_f16, x, total_rows, K, offsets, E, codes, scales,
                      scale_row_offsets);
}

/* Step 6 with the MoE dispatch gather in front ([PR43557] item 3: the
 * experts-quant input is the routed, expert-sorted activations): output row r
 * is source row row_index[r]; out-of-range indices give zero rows and -7.
 * Plainly: gather the rows, then the grouped quantize above. */
static int gather_with(dense_quantize_fn quantize, const uint16_t* x, int64_t num_src_rows,
                       int64_t K, int64_t ldx, const int32_t* row_index, int64_t total_rows,
                       const int32_t* offsets, int32_t E, uint8_t* codes, uint8_t* scales,
                       int32_t* scale_row_offsets) {
  uint16_t* g = (uint16_t*)calloc((size_t)(total_rows * K) + 1, sizeof(uint16_t));
  int bad = 0;
  for (int64_t r = 0; r < total_rows; ++r) {
    int64_t src = row_index[r];
    if (src < 0 || src >= num_src_rows) {
      bad = 1;
      continue; /* stays a zero row */
    }
    memcpy(g + r * K, x + src * ldx, (size_t)K * sizeof(uint16_t));
  }
  int rc = grouped_with(quantize, g, total_rows, K, offsets, E, codes, scales, scale_row_offsets);
  free(g);
  if (rc != 0) return rc;
  return bad ? -7 : 0;
}

int orc_quantize_grouped_gather(const uint16_t* x, int64_t num_src_rows, int64_t K, int64_t ldx,
                                const int32_t* row_index, int64_t total_rows,
                                const int32_t* offsets, int32_t E, uint8_t* codes,
                                uint8_t* scales, int32_t* scale_row_offsets) {
  return gather_with(orc_quantize, x, num_src_rows, K, ldx, row_index, total_rows, offsets, E,
                     codes, scales, scale_row_offsets);
}

int orc_quantize_grouped_gather_f16(const uint16_t* x, int64_t num_src_rows, int64_t K,
                                    int64_t ldx, const int32_t* row_index, int64_t total_rows,
                                    const int32_t* offsets, int32_t E, uint8_t* codes,
                                    uint8_t* scales, int32_t* scale_row_offsets) {
  return gather_with(orc_quantize_f16, x, num_src_rows, K, ldx, row_index, total_rows, offsets, E,
                     codes, scales, scale_row_offsets);
}

/* Step 6 with the MoE dispatch as a scatter ([PR43557] item 3: the
 * experts-quant input is the routed, expert-sorted activations), in the form a
 * router's sort produces: route j of token t lands on row
 * dest_rows[t * top_k + j] of the expert-sorted batch, -1 meaning the route is
 * not dispatched.  Plainly: place every token row on its destination rows,
 * run the grouped quantize above on that batch, then keep the rows some route
 * targets (their codes and the scale bytes of their padded rows) and every
 * segment's pad rows (zero scale bytes); rows no route targets are left as
 * they were.  An entry outside [-1, total_rows) is skipped and gives -7; bad
 * offsets give -6 and nothing is written but the -1 scale row offsets. */
static int scatter_with(dense_quantize_fn quantize, const uint16_t* x, int64_t num_tokens,
                        int64_t K, int64_t ldx, const int32_t* dest_rows, int32_t top_k,
                        int64_t total_rows, const int32_t* offsets, int32_t E, uint8_t* codes,
                        uint8_t* scales, int32_t* scale_row_offsets) {
  int bad = 0;
  uint16_t* g = (uint16_t*)calloc((size_t)(total_rows * K) + 1, sizeof(uint16_t));
  uint8_t* hit = (uint8_t*)calloc((size_t)total_rows + 1, 1);
  for (int64_t t = 0; t < num_tokens; ++t)
    for (int32_t j = 0; j < top_k; ++j) {
      int64_t d = dest_rows[t * top_k + j];
      if (d == -1) continue;
      if (d < -1 || d >= total_rows) {
        bad = 1;
        continue;
      }
      memcpy(g + d * K, x + t * ldx, (size_t)K * sizeof(uint16_t));
      hit[d] = 1;
    }
  int64_t sK = K / 32;
  int64_t nkt = (sK + 3) / 4;
  int64_t padded_sK = nkt * 4;
  /* the segments' padded rows never exceed total_rows + 127 E */
  int64_t bound_rows = (total_rows + 127 * (int64_t)(E > 0 ? E : 0)) / 128 * 128 + 128;
  uint8_t* tc = (uint8_t*)calloc((size_t)(total_rows * (K / 2)) + 1, 1);
  uint8_t* ts = (uint8_t*)calloc((size_t)(bound_rows * padded_sK) + 1, 1);
  int rc = grouped_with(quantize, g, total_rows, K, offsets, E, tc, ts, scale_row_offsets);
  if (rc == 0) {
    for (int32_t e = 0; e < E; ++e) {
      int64_t n = (int64_t)offsets[e + 1] - offsets[e];
      int64_t base = (int64_t)scale_row_offsets[e] * padded_sK;
      for (int64_t prow = 0; prow < (n + 127) / 128 * 128; ++prow) {
        int64_t d = offsets[e] + prow;
        if (prow < n && !hit[d]) continue; /* untargeted: left as it was */
        if (prow < n) memcpy(codes + d * (K / 2), tc + d * (K / 2), (size_t)(K / 2));
        for (int64_t c = 0; c < padded_sK; ++c) {
          int64_t i = base + tiled_index(prow, c, nkt);
          scales[i] = ts[i];
        }
      }
    }
  }
  free(g);
  free(hit);
  free(tc);
  free(ts);
  if (rc != 0) return rc;
  return bad ? -7 : 0;
}

int orc_quantize_grouped_scatter(const uint16_t* x, int64_t num_tokens, int64_t K, int64_t ldx,
                                 const int32_t* dest_rows, int32_t top_k, int64_t total_rows,
                                 const int32_t* offsets, int32_t E, uint8_t* codes,
                                 uint8_t* scales, int32_t* scale_row_offsets) {
  return scatter_with(orc_quantize, x, num_tokens, K, ldx, dest_rows, top_k, total_rows, offsets,
                      E, codes, scales, scale_row_offsets);
}

int orc_quantize_grouped_scatter_f16(const uint16_t* x, int64_t num_tokens, int64_t K,
                                     int64_t ldx, const int32_t* dest_rows, int32_t top_k,
                                     int64_t total_rows, const int32_t* offsets, int32_t E,
                                     uint8_t* codes, uint8_t* scales,
                                     int32_t* scale_row_offsets) {
  return scatter_with(orc_quantize_f16, x, num_tokens, K, ldx, dest_rows, top_k, total_rows,
                      offsets, E, codes, scales, scale_row_offsets);
}

/* Step 7 — dequantize: for each element, its nibble and its block's scale
 * byte (read back through the tiled layout) give E2M1 value * 2^(s-127),
 * rounded once to BF16.  [PR46915] "Motivation" (FP4 -> BF16 table);
 * [PR43557] excerpt (scale value from the exponent bits). */
void orc_dequantize(const uint8_t* codes, const uint8_t* tiled_scales,
                    int64_t M, int64_t K, uint16_t* y) {
  int64_t sK = K / 32;
  if (M <= 0 || sK <= 0) return;
  uint8_t* flat = (uint8_t*)calloc((size_t)(M * sK), 1);
  orc_untile_scales(tiled_scales, M, sK, flat);
  for (int64_t r = 0; r < M; ++r)
    for (int64_t k = 0; k < K; ++k) {
      uint8_t byte = codes[r * (K / 2) + k / 2];
      uint8_t nib = (k % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
      y[r * K + k] = dequant_value(nib, flat[r * sK + k / 32]);
    }
  free(flat);
}

/* Step 8 — [w1; w3] -> [w3; w1].  [PR51038] "Implementation breakdown"
 * item 2 and the convert_weight_to_mxfp4_moe_kernel_format branch: the two
 * halves of dim 1 (2N rows per expert) of the w13 codes and scales change
 * places; the w13 bias is cut in two along its last dim, re-joined as
 * [b3, b1] and cast to BF16; the w2 bias is only cast to BF16.  Tiled scales
 * are swapped by logical row: untile, swap, tile. */
void orc_swap_halves(const uint8_t* in, uint8_t* out, int64_t E, int64_t two_n,
                     int64_t row_bytes) {
  int64_t n = two_n / 2;
  for (int64_t e = 0; e < E; ++e)
    for (int64_t r = 0; r < two_n; ++r)
      memcpy(out + (e * two_n + r) * row_bytes, in + (e * two_n + (r + n) % two_n) * row_bytes,
             (size_t)row_bytes);
}

void orc_swap_bias_bf16(const float* in, uint16_t* out, int64_t E, int64_t two_n) {
  int64_t n = two_n / 2;
  for (int64_t e = 0; e < E; ++e)
    for (int64_t j = 0; j < two_n; ++j) /* [b1, b3] -> [b3, b1], then BF16 */
      out[e * two_n + j] = orc_double_to_bf16_rne((double)in[e * two_n + (j + n) % two_n]);
}

void orc_cast_bf16(const float* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_double_to_bf16_rne((double)in[i]);
}

void orc_swap_w13(const uint8_t* codes_in, const uint8_t* scales_in,
                  const float* w13_bias_in, int32_t E, int64_t two_n, int64_t K,
                  int32_t scales_tiled, uint8_t* codes_out, uint8_t* scales_out,
                  uint16_t* w13_bias_out, const float* w2_bias_in,
                  int64_t w2_bias_numel, uint16_t* w2_bias_out) {
  int64_t sK = K / 32;
  size_t tiled_bytes = orc_scale_bytes(two_n, K);
  orc_swap_halves(codes_in, codes_out, E, two_n, K / 2);
  if (scales_tiled) {
    uint8_t* flat_in = (uint8_t*)calloc((size_t)(two_n * sK) + 1, 1);
    uint8_t* flat_out = (uint8_t*)calloc((size_t)(two_n * sK) + 1, 1);
    for (int32_t e = 0; e < E; ++e) {
      orc_untile_scales(scales_in + e * tiled_bytes, two_n, sK, flat_in);
      orc_swap_halves(flat_in, flat_out, 1, two_n, sK);
      orc_tile_scales(flat_out, two_n, sK, scales_out + e * tiled_bytes);
    }
    free(flat_in);
    free(flat_out);
  } else {
    orc_swap_halves(scales_in, scales_out, E, two_n, sK);
  }
  if (w13_bias_in) orc_swap_bias_bf16(w13_bias_in, w13_bias_out, E, two_n);
  if (w2_bias_in) orc_cast_bf16(w2_bias_in, w2_bias_out, w2_bias_numel);
}

/* ======================================================================
 * NVFP4 — the other branch of the pages' quantize kernel ([PR43557]
 * "Implementation breakdown" item 1, the non-UE8M0 branch of the
 * cvt_warp_fp16_to_fp4 excerpt, and "Review highlights": the block scale is
 * SFScaleVal * vecMax / 6 stored as FP8 E4M3, and the value used to scale the
 * elements must be the E4M3-rounded one, SFValue = float(E4M3 byte)).
 * Readings where the pages are silent: 16-element blocks; the global scale
 * SFScaleVal (g) is a float supplied by the caller; every step is one IEEE
 * float32 operation rounded to nearest even, in this order:
 *   q   = vecMax / 6;  sf = g * q;  byte = E4M3_RNE_satfinite(sf);
 *   SFValue = float(byte);  inv = g / SFValue;  y = x * inv;
 *   code = E2M1 RNE (saturating) of y;  blocks with byte == 0 emit 0x0.
 * Dequantize: t = e2m1(code) * SFValue (exact); y = t * (1/g) with 1/g one
 * float32 division, as NVFP4 consumers apply one global dequant factor;
 * BF16 RNE of y.
 * ====================================================================== */

/* FP8 E4M3 (OCP FP8, "fn" variant): sign, 4-bit exponent (bias 7), 3-bit
 * mantissa, exponent 0 subnormal (m * 2^-9), largest finite 448 (0x7E), 0x7F
 * NaN, no infinities. */
double orc_e4m3_to_double(uint8_t b) {
  int sign = (b >> 7) & 1;
  int e = (b >> 3) & 0xF;
  int m = b & 7;
  double v;
  if (e == 15 && m == 7) v = NAN;
  else if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp(8.0 + m, e - 10);
  return sign ? -v : v;
}

/* Nearest E4M3 value, ties to the even mantissa, magnitudes above 448
 * saturate to 448 (satfinite); NaN -> 0x7F. */
uint8_t orc_e4m3_from_double(double d) {
  uint8_t sign = signbit(d) ? 0x80u : 0u;
  if (isnan(d)) return (uint8_t)(sign | 0x7Fu);
  double a = fabs(d);
  if (a >= 448.0) return (uint8_t)(sign | 0x7Eu);
  /* quantum: 2^-9 in the subnormal range (a < 2^-6), else 2^(e-3) */
  int e;
  frexp(a, &e);
  int ex = e - 1; /* floor(log2 a) */
  int qexp = (a < ldexp(1.0, -6)) ? -9 : ex - 3;
  double n = nearbyint(ldexp(a, -qexp));
  double r = ldexp(n, qexp);
  if (r > 448.0) r = 448.0;
  if (r == 0.0) return sign;
  if (r < ldexp(1.0, -6)) return (uint8_t)(sign | (uint8_t)n); /* subnormal */
  frexp(r, &e);
  int rexp = e - 1;
  uint32_t mant = (uint32_t)(ldexp(r, -rexp) * 8.0 - 8.0);
  return (uint8_t)(sign | ((uint32_t)(rexp + 7) << 3) | mant);
}

static float f32_of_bf16(uint16_t b) { return bf16_to_float(b); }

/* Steps of one 16-element block: its E4M3 scale byte and 16 nibbles. */
/* A 16-bit element as float (exact for both input formats). */
static float f32_of_f16(uint16_t h) { return (float)orc_f16_to_double(h); }
typedef float (*to_f32_fn)(uint16_t);

static void nvfp4_block_of(to_f32_fn to_f32, const uint16_t* x, float g, uint8_t* sf_byte,
                           uint8_t* nib) {
  float vmax = 0.0f;
  for (int i = 0; i < 16; ++i) {
    float a = to_f32((uint16_t)(x[i] & 0x7FFFu));
    if (a > vmax) vmax = a;
  }
  float q = vmax / 6.0f; /* each float step rounds once (no contraction) */
  float sf = g * q;
  uint8_t byte = orc_e4m3_from_double((double)sf);
  *sf_byte = byte;
  float sfv = (float)orc_e4m3_to_double(byte);
  if (byte == 0 || sfv == 0.0f) {
    for (int i = 0; i < 16; ++i) nib[i] = 0;
    return;
  }
  float inv = g / sfv;
  for (int i = 0; i < 16; ++i) {
    float y = to_f32(x[i]) * inv;
    nib[i] = e2m1_round((double)y, (x[i] >> 15) & 1u);
  }
}

size_t orc_nvfp4_scale_bytes(int64_t M, int64_t K) {
  if (M <= 0 || K <= 0 || K % 16 != 0) return 0;
  return (size_t)((M + 127) / 128 * 128 * ((K / 16 + 3) / 4 * 4));
}

static void nvfp4_flat_of(to_f32_fn to_f32, const uint16_t* x, int64_t M, int64_t K, int64_t ldx,
                          float g, uint8_t* codes, uint8_t* flat_scales) {
  int64_t sK = K / 16;
  for (int64_t r = 0; r < M; ++r)
    for (int64_t b = 0; b < sK; ++b) {
      uint8_t nib[16];
      nvfp4_block_of(to_f32, x + r * ldx + b * 16, g, &flat_scales[r * sK + b], nib);
      for (int j = 0; j < 8; ++j)
        codes[r * (K / 2) + b * 8 + j] = (uint8_t)(nib[2 * j] | (nib[2 * j + 1] << 4));
    }
}

void orc_nvfp4_quantize_flat(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, float g,
                             uint8_t* codes, uint8_t* flat_scales) {
  nvfp4_flat_of(f32_of_bf16, x, M, K, ldx, g, codes, flat_scales);
}

static void nvfp4_quantize_of(to_f32_fn to_f32, const uint16_t* x, int64_t M, int64_t K,
                              int64_t ldx, float g, uint8_t* codes, uint8_t* tiled_scales) {
  int64_t sK = K / 16;
  if (M <= 0 || sK <= 0) return;
  uint8_t* flat = (uint8_t*)calloc((size_t)(M * sK), 1);
  nvfp4_flat_of(to_f32, x, M, K, ldx, g, codes, flat);
  orc_tile_scales(flat, M, sK, tiled_scales); /* same 128x4 tiling, 16-element columns */
  free(flat);
}

void orc_nvfp4_quantize(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, float g,
                        uint8_t* codes, uint8_t* tiled_scales) {
  nvfp4_quantize_of(f32_of_bf16, x, M, K, ldx, g, codes, tiled_scales);
}

/* The same NVFP4 steps on IEEE binary16 input (every FP16 value is exact in
 * float32, so only the decoding of the element changes). */
void orc_nvfp4_quantize_f16(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, float g,
                            uint8_t* codes, uint8_t* tiled_scales) {
  nvfp4_quantize_of(f32_of_f16, x, M, K, ldx, g, codes, tiled_scales);
}

/* NVFP4 experts quant: the grouped layout of step 6 with the NVFP4 block
 * ([PR43557] item 3 names the experts-quant kernel, whose non-UE8M0 branch is
 * the NVFP4 one).  Segment e = rows [o[e], o[e+1]) is quantized as its own
 * matrix with its own global scale g[e]; codes keep the row order; its tiled
 * E4M3 scales (16-element columns, padded to 128 rows) start at padded row
 * P[e].  Bad offsets: -6, scale row offsets all -1, nothing else written. */
static int nvfp4_grouped_of(to_f32_fn to_f32, const uint16_t* x, int64_t total_rows, int64_t K,
                            const int32_t* offsets, int32_t E, const float* g, uint8_t* codes,
                            uint8_t* scales, int32_t* scale_row_offsets) {
  int ok = (E >= 0) && offsets[0] == 0 && (int64_t)offsets[E] == total_rows;
  for (int32_t e = 0; ok && e < E; ++e) ok = offsets[e] <= offsets[e + 1];
  if (!ok) {
    for (int32_t e = 0; e <= E; ++e) scale_row_offsets[e] = -1;
    return -6;
  }
  int64_t padded_sK = (K / 16 + 3) / 4 * 4;
  int64_t P = 0;
  for (int32_t e = 0; e < E; ++e) {
    int64_t n = (int64_t)offsets[e + 1] - offsets[e];
    scale_row_offsets[e] = (int32_t)P;
    nvfp4_quantize_of(to_f32, x + (int64_t)offsets[e] * K, n, K, K, g[e],
                      codes + (int64_t)offsets[e] * (K / 2), scales + P * padded_sK);
    P += (n + 127) / 128 * 128;
  }
  scale_row_offsets[E] = (int32_t)P;
  return 0;
}

int orc_nvfp4_quantize_grouped(const uint16_t* x, int64_t total_rows, int64_t K,
                               const int32_t* offsets, int32_t E, const float* g,
                               uint8_t* codes, uint8_t* scales, int32_t* scale_row_offsets) {
  return nvfp4_grouped_of(f32_of_bf16, x, total_rows, K, offsets, E, g, codes, scales,
                          scale_row_offsets);
}

int orc_nvfp4_quantize_grouped_f16(const uint16_t* x, int64_t total_rows, int64_t K,
                                   const int32_t* offsets, int32_t E, const float* g,
                                   uint8_t* codes, uint8_t* scales, int32_t* scale_row_offsets) {
  return nvfp4_grouped_of(f32_of_f16, x, total_rows, K, offsets, E, g, codes, scales,
                          scale_row_offsets);
}

/* NVFP4 experts quant with the dispatch as a scatter: route j of token t
 * lands on row dest_rows[t * top_k + j] of the expert-sorted batch (-1: not
 * dispatched).  The result is the NVFP4 experts quant above of the batch the
 * routes fill, each expert segment with its own global scale g[e]; rows that
 * no route targets keep their bytes (codes and scales), pad rows get zero
 * scales.  Entries outside [-1, total_rows) are skipped (-7); bad offsets as
 * in the experts quant (-6). */
static int nvfp4_scatter_of(to_f32_fn to_f32, const uint16_t* x, int64_t num_tokens, int64_t K,
                            int64_t ldx, const int32_t* dest_rows, int32_t top_k,
                            int64_t total_rows, const int32_t* offsets, int32_t E,
                            const float* g, uint8_t* codes, uint8_t* scales,
                            int32_t* scale_row_offsets) {
  int bad = 0;
  uint16_t* batch = (uint16_t*)calloc((size_t)(total_rows * K) + 1, sizeof(uint16_t));
  uint8_t* hit = (uint8_t*)calloc((size_t)total_rows + 1, 1);
  for (int64_t t = 0; t < num_tokens; ++t)
    for (int32_t j = 0; j < top_k; ++j) {
      int64_t d = dest_rows[t * top_k + j];
      if (d == -1) continue;
      if (d < -1 || d >= total_rows) {
        bad = 1;
        continue;
      }
      memcpy(batch + d * K, x + t * ldx, (size_t)K * sizeof(uint16_t));
      hit[d] = 1;
    }
  int64_t nkt = (K / 16 + 3) / 4;
  int64_t padded_sK = nkt * 4;
  int64_t bound_rows = (total_rows + 127 * (int64_t)(E > 0 ? E : 0)) / 128 * 128 + 128;
  uint8_t* tc = (uint8_t*)calloc((size_t)(total_rows * (K / 2)) + 1, 1);
  uint8_t* ts = (uint8_t*)calloc((size_t)(bound_rows * padded_sK) + 1, 1);
  int rc = nvfp4_grouped_of(to_f32, batch, total_rows, K, offsets, E, g, tc, ts,
                            scale_row_offsets);
  if (rc == 0) {
    for (int32_t e = 0; e < E; ++e) {
      int64_t n = (int64_t)offsets[e + 1] - offsets[e];
      int64_t base = (int64_t)scale_row_offsets[e] * padded_sK;
      for (int64_t prow = 0; prow < (n + 127) / 128 * 128; ++prow) {
        int64_t d = offsets[e] + prow;
        if (prow < n && !hit[d]) continue; /* untargeted: left as it was */
        if (prow < n) memcpy(codes + d * (K / 2), tc + d * (K / 2), (size_t)(K / 2));
        for (int64_t c = 0; c < padded_sK; ++c) {
          int64_t i = base + tiled_index(prow, c, nkt);
          scales[i] = ts[i];
        }
      }
    }
  }
  free(batch);
  free(hit);
  free(tc);
  free(ts);
  if (rc != 0) return rc;
  return bad ? -7 : 0;
}

int orc_nvfp4_quantize_grouped_scatter(const uint16_t* x, int64_t num_tokens, int64_t K,
                                       int64_t ldx, const int32_t* dest_rows, int32_t top_k,
                                       int64_t total_rows, const int32_t* offsets, int32_t E,
                                       const float* g, uint8_t* codes, uint8_t* scales,
                                       int32_t* scale_row_offsets) {
  return nvfp4_scatter_of(f32_of_bf16, x, num_tokens, K, ldx, dest_rows, top_k, total_rows,
                          offsets, E, g, codes, scales, scale_row_offsets);
}

int orc_nvfp4_quantize_grouped_scatter_f16(const uint16_t* x, int64_t num_tokens, int64_t K,
                                           int64_t ldx, const int32_t* dest_rows, int32_t top_k,
                                           int64_t total_rows, const int32_t* offsets, int32_t E,
                                           const float* g, uint8_t* codes, uint8_t* scales,
                                           int32_t* scale_row_offsets) {
  return nvfp4_scatter_of(f32_of_f16, x, num_tokens, K, ldx, dest_rows, top_k, total_rows,
                          offsets, E, g, codes, scales, scale_row_offsets);
}

void orc_nvfp4_dequantize(const uint8_t* codes, const uint8_t* tiled_scales, int64_t M, int64_t K,
                          float g, uint16_t* y) {
  int64_t sK = K / 16;
  if (M <= 0 || sK <= 0) return;
  uint8_t* flat = (uint8_t*)calloc((size_t)(M * sK), 1);
  orc_untile_scales(tiled_scales, M, sK, flat);
  float inv_g = 1.0f / g;
  for (int64_t r = 0; r < M; ++r)
    for (int64_t k = 0; k < K; ++k) {
      uint8_t byte = codes[r * (K / 2) + k / 2];
      uint8_t nib = (k % 2 == 0) ? (byte & 0xFu) : (byte >> 4);
      uint8_t sb = flat[r * sK + k / 16];
      if ((sb & 0x7Fu) == 0x7Fu) { /* the E4M3 NaN: the canonical BF16 NaN, as E8M0 255 */
        y[r * K + k] = 0x7FC0u;
        continue;
      }
      float sfv = (float)orc_e4m3_to_double(sb);
      float t = (float)orc_e2m1_decode(nib) * sfv; /* exact */
      float v = t * inv_g;
      y[r * K + k] = orc_double_to_bf16_rne((double)v);
    }
  free(flat);
}

void orc_e4m3_from_double_many(const double* d, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_from_double(d[i]);
}

/* The MoE dispatch permutation from the router's choices ([PR43557]
 * "Implementation breakdown" item 3: the experts quant takes the routed
 * activations sorted by expert; this is the sort).  Entry i = t * top_k + j
 * of topk_ids is expert topk_ids[i] of route j of token t.  Rows are the
 * entries with a valid expert (0 <= id < E) in order of expert, then of i;
 * offsets[e] is the first row of expert e, offsets[E] the number of rows;
 * dest_rows[i] is the row of entry i (-1 for an entry not dispatched) and
 * row_index[row] its token (may be NULL).  Returns 0, or -7 when some id is
 * neither -1 (not dispatched) nor in [0, E). */
int orc_moe_route(const int32_t* topk_ids, int64_t num_tokens, int32_t top_k, int32_t E,
                  int32_t* offsets, int32_t* dest_rows, int32_t* row_index) {
  const int64_t n = num_tokens * top_k;
  int bad = 0;
  for (int64_t i = 0; i < n; ++i) {
    dest_rows[i] = -1;
    if (topk_ids[i] != -1 && (topk_ids[i] < 0 || topk_ids[i] >= E)) bad = 1;
  }
  int64_t row = 0;
  for (int32_t e = 0; e < E; ++e) {
    offsets[e] = (int32_t)row;
    for (int64_t i = 0; i < n; ++i)
      if (topk_ids[i] == e) {
        dest_rows[i] = (int32_t)row;
        if (row_index != NULL) row_index[row] = (int32_t)(i / top_k);
        ++row;
      }
  }
  offsets[E] = (int32_t)row;
  return bad ? -7 : 0;
}
