/* A plain C caller of libmxfp4_gb300.so against the CPU oracle (test
 * infrastructure, linked into this test program only): a small MoE batch
 * (300 tokens, top-4 over 13 experts, K = 2880, so partial k-tiles and
 * ragged segments) through the dispatch calls in both directions, the dense
 * quantize and dequantize, the NVFP4 experts quant as a scatter and the w13
 * swap, every output byte compared.  Inputs are BF16 bit patterns drawn from
 * a fixed counter-based stream (no arithmetic of the method).  Exit status 0
 * when every call matches. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "mxfp4.h"
#include "mxfp4_oracle.h"

enum { T = 300, TOPK = 4, E = 13, K = 2880, R = T * TOPK };

#define CHECK_CUDA(call)                                                    \
  do {                                                                      \
    cudaError_t e_ = (call);                                                \
    if (e_ != cudaSuccess) {                                                \
      fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));           \
      exit(2);                                                              \
    }                                                                       \
  } while (0)

#define CHECK_RC(call)                                                      \
  do {                                                                      \
    int r_ = (call);                                                        \
    if (r_ != MXFP4_OK) {                                                   \
      fprintf(stderr, "%s: %s\n", #call, mxfp4_status_string(r_));          \
      exit(1);                                                              \
    }                                                                       \
  } while (0)

static uint64_t g_state = 0x9E3779B97F4A7C15ull;

/* splitmix64 */
static uint64_t next_u64(void) {
  uint64_t z = (g_state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* A BF16 pattern with a random sign, a biased exponent in [117, 136] and a
 * random 7-bit mantissa (magnitudes 2^-10 .. 2^10). */
static uint16_t next_bf16(void) {
  const uint64_t r = next_u64();
  const uint16_t sign = (uint16_t)((r & 1u) << 15);
  const uint16_t ex = (uint16_t)(117u + (r >> 8) % 20u);
  return (uint16_t)(sign | (ex << 7) | ((r >> 32) & 0x7Fu));
}

static void* dev_copy(const void* h, size_t n) {
  void* d = NULL;
  CHECK_CUDA(cudaMalloc(&d, n > 0 ? n : 1));
  if (n > 0) CHECK_CUDA(cudaMemcpy(d, h, n, cudaMemcpyHostToDevice));
  return d;
}

static void* dev_fill(size_t n, int byte) {
  void* d = NULL;
  CHECK_CUDA(cudaMalloc(&d, n > 0 ? n : 1));
  CHECK_CUDA(cudaMemset(d, byte, n > 0 ? n : 1));
  return d;
}

static int same(const char* what, const void* dev, const void* want, size_t n) {
  unsigned char* h = (unsigned char*)malloc(n > 0 ? n : 1);
  CHECK_CUDA(cudaMemcpy(h, dev, n, cudaMemcpyDeviceToHost));
  const unsigned char* w = (const unsigned char*)want;
  for (size_t i = 0; i < n; ++i)
    if (h[i] != w[i]) {
      fprintf(stderr, "%s: byte %zu is 0x%02x, oracle 0x%02x\n", what, i, h[i], w[i]);
      free(h);
      return 0;
    }
  free(h);
  return 1;
}

int main(void) {
  static uint16_t x[T * K];
  for (int i = 0; i < T * K; ++i) x[i] = next_bf16();
  /* route j of token t: expert (t + j * (1 + t % 12)) % 13, distinct for j < 4 */
  static int32_t expert[T][TOPK], dest[T][TOPK], row_index[R], off[E + 1];
  for (int t = 0; t < T; ++t)
    for (int j = 0; j < TOPK; ++j) expert[t][j] = (t + j * (1 + t % 12)) % E;
  int row = 0;
  for (int e = 0; e < E; ++e) {
    off[e] = row;
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < TOPK; ++j)
        if (expert[t][j] == e) {
          dest[t][j] = row;
          row_index[row++] = t;
        }
  }
  off[E] = row;

  const size_t code_bytes = (size_t)R * (K / 2);
  const size_t bound = mxfp4_grouped_scale_bytes_bound(R, E, K);
  uint8_t* codes_o = (uint8_t*)calloc(code_bytes, 1);
  uint8_t* scales_o = (uint8_t*)calloc(bound, 1);
  int32_t sro_o[E + 1];
  if (orc_quantize_grouped_gather(x, T, K, K, row_index, R, off, E, codes_o, scales_o, sro_o) != 0)
    return 1;
  const size_t used = (size_t)sro_o[E] * ((K / 32 + 3) / 4 * 4);

  void* dx = dev_copy(x, sizeof x);
  void* ddest = dev_copy(dest, sizeof dest);
  void* drow = dev_copy(row_index, sizeof row_index);
  void* doff = dev_copy(off, sizeof off);
  int ok = 1;

  /* the dispatch as a scatter with a workspace, and as a gather without one */
  {
    const size_t ws_bytes = mxfp4_scatter_workspace_bytes(T, R, E, K);
    void* ws = dev_fill(ws_bytes, 0x5A);
    void* dc = dev_fill(code_bytes, 0xA5);
    void* ds = dev_fill(bound, 0xA5);
    void* dsro = dev_fill(sizeof sro_o, 0xA5);
    void* dst = dev_fill(4, 0xA5);
    CHECK_RC(mxfp4_quantize_grouped_scatter_ws(dx, T, K, K, (const int32_t*)ddest, TOPK, R,
                                               (const int32_t*)doff, E, ws, ws_bytes,
                                               (uint8_t*)dc, (uint8_t*)ds, (int32_t*)dsro,
                                               (int32_t*)dst, NULL));
    const int32_t zero = 0;
    ok &= same("scatter status", dst, &zero, 4) && same("scatter offsets", dsro, sro_o,
                                                         sizeof sro_o);
    ok &= same("scatter codes", dc, codes_o, code_bytes) &&
          same("scatter scales", ds, scales_o, used);
    CHECK_CUDA(cudaMemset(dc, 0xA5, code_bytes));
    CHECK_CUDA(cudaMemset(ds, 0xA5, bound));
    CHECK_RC(mxfp4_quantize_grouped_gather(dx, T, K, K, (const int32_t*)drow, R,
                                           (const int32_t*)doff, E, (uint8_t*)dc, (uint8_t*)ds,
                                           (int32_t*)dsro, (int32_t*)dst, NULL));
    ok &= same("gather status", dst, &zero, 4) && same("gather offsets", dsro, sro_o,
                                                       sizeof sro_o);
    ok &= same("gather codes", dc, codes_o, code_bytes) &&
          same("gather scales", ds, scales_o, used);
    cudaFree(ws);
    cudaFree(dc);
    cudaFree(ds);
    cudaFree(dsro);
    cudaFree(dst);
  }

  /* dense quantize of the token rows, then dequantize */
  {
    const size_t cb = (size_t)T * (K / 2), sb = mxfp4_scale_bytes(T, K);
    uint8_t* c = (uint8_t*)calloc(cb, 1);
    uint8_t* s = (uint8_t*)calloc(sb, 1);
    uint16_t* y = (uint16_t*)calloc((size_t)T * K, 2);
    orc_quantize(x, T, K, K, c, s);
    orc_dequantize(c, s, T, K, y);
    void* dc = dev_fill(cb, 0);
    void* ds = dev_fill(sb, 0);
    void* dy = dev_fill((size_t)T * K * 2, 0);
    CHECK_RC(mxfp4_quantize(dx, T, K, K, (uint8_t*)dc, (uint8_t*)ds, NULL));
    CHECK_RC(mxfp4_dequantize((const uint8_t*)dc, (const uint8_t*)ds, T, K, dy, NULL));
    ok &= same("dense codes", dc, c, cb) && same("dense scales", ds, s, sb) &&
          same("dequantized", dy, y, (size_t)T * K * 2);
    cudaFree(dc);
    cudaFree(ds);
    cudaFree(dy);
    free(c);
    free(s);
    free(y);
  }

  /* NVFP4 experts quant with the dispatch as a scatter, a global scale per expert */
  {
    float gs[E];
    for (int e = 0; e < E; ++e) gs[e] = 448.0f * 6.0f / (float)(1 + e * 37);
    const size_t nb = mxfp4_nvfp4_grouped_scale_bytes_bound(R, E, K);
    uint8_t* c = (uint8_t*)calloc(code_bytes, 1);
    uint8_t* s = (uint8_t*)calloc(nb, 1);
    int32_t sro[E + 1];
    if (orc_nvfp4_quantize_grouped_scatter(x, T, K, K, &dest[0][0], TOPK, R, off, E, gs, c, s,
                                           sro) != 0)
      return 1;
    const size_t nused = (size_t)sro[E] * ((K / 16 + 3) / 4 * 4);
    const size_t ws_bytes = mxfp4_nvfp4_scatter_workspace_bytes(R, E, K);
    void* ws = dev_fill(ws_bytes, 0x5A);
    void* dg = dev_copy(gs, sizeof gs);
    void* dc = dev_fill(code_bytes, 0);
    void* ds = dev_fill(nb, 0);
    void* dsro = dev_fill(sizeof sro, 0);
    CHECK_RC(mxfp4_quantize_nvfp4_grouped_scatter_ws(dx, T, K, K, (const int32_t*)ddest, TOPK,
                                                     R, (const int32_t*)doff, E,
                                                     (const float*)dg, ws, ws_bytes,
                                                     (uint8_t*)dc, (uint8_t*)ds, (int32_t*)dsro,
                                                     NULL, NULL));
    ok &= same("nvfp4 offsets", dsro, sro, sizeof sro) && same("nvfp4 codes", dc, c, code_bytes) &&
          same("nvfp4 scales", ds, s, nused);
    cudaFree(ws);
    cudaFree(dg);
    cudaFree(dc);
    cudaFree(ds);
    cudaFree(dsro);
    free(c);
    free(s);
  }

  /* w13 swap: 3 experts, 2N = 150 (N odd), flat scales, both biases */
  {
    enum { SE = 3, TWO_N = 150, SK = 256, W2N = 37 };
    static uint8_t c_in[SE * TWO_N * (SK / 2)], s_in[SE * TWO_N * (SK / 32)];
    static float b13[SE * TWO_N], b2[SE * W2N];
    for (size_t i = 0; i < sizeof c_in; ++i) c_in[i] = (uint8_t)next_u64();
    for (size_t i = 0; i < sizeof s_in; ++i) s_in[i] = (uint8_t)next_u64();
    for (int i = 0; i < SE * TWO_N; ++i) {
      const uint32_t b = (uint32_t)next_bf16() << 16 | (uint32_t)(next_u64() & 0xFFFFu);
      memcpy(&b13[i], &b, 4);
    }
    for (int i = 0; i < SE * W2N; ++i) {
      const uint32_t b = (uint32_t)next_bf16() << 16 | (uint32_t)(next_u64() & 0xFFFFu);
      memcpy(&b2[i], &b, 4);
    }
    static uint8_t c_o[sizeof c_in], s_o[sizeof s_in];
    static uint16_t b13_o[SE * TWO_N], b2_o[SE * W2N];
    orc_swap_w13(c_in, s_in, b13, SE, TWO_N, SK, 0, c_o, s_o, b13_o, b2, SE * W2N, b2_o);
    void* dci = dev_copy(c_in, sizeof c_in);
    void* dsi = dev_copy(s_in, sizeof s_in);
    void* db13 = dev_copy(b13, sizeof b13);
    void* db2 = dev_copy(b2, sizeof b2);
    void* dco = dev_fill(sizeof c_in, 0);
    void* dso = dev_fill(sizeof s_in, 0);
    void* db13o = dev_fill(sizeof b13_o, 0);
    void* db2o = dev_fill(sizeof b2_o, 0);
    CHECK_RC(mxfp4_swap_w13((const uint8_t*)dci, (const uint8_t*)dsi, (const float*)db13, SE,
                            TWO_N, SK, 0, (uint8_t*)dco, (uint8_t*)dso, db13o,
                            (const float*)db2, SE * W2N, db2o, NULL));
    ok &= same("swapped codes", dco, c_o, sizeof c_o) &&
          same("swapped scales", dso, s_o, sizeof s_o) &&
          same("w13 bias", db13o, b13_o, sizeof b13_o) && same("w2 bias", db2o, b2_o,
                                                               sizeof b2_o);
    cudaFree(dci);
    cudaFree(dsi);
    cudaFree(db13);
    cudaFree(db2);
    cudaFree(dco);
    cudaFree(dso);
    cudaFree(db13o);
    cudaFree(db2o);
  }

  CHECK_CUDA(cudaDeviceSynchronize());
  cudaFree(dx);
  cudaFree(ddest);
  cudaFree(drow);
  cudaFree(doff);
  free(codes_o);
  free(scales_o);
  if (!ok) return 1;
  printf("c abi: scatter, gather, dense, dequantize, NVFP4 scatter and swap match the oracle\n");
  return 0;
}
