/* A plain C caller of libmxfp4_gb300.so: quantizes one 1 x 32 BF16 block whose
 * expected codes and scale were derived by hand (vecMax 1.5 -> scale exponent
 * 125; every E2M1 tie point), dequantizes it, and checks every byte.
 * Exit status 0 on success. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <cuda_runtime.h>

#include "mxfp4.h"

#define CHECK_CUDA(call)                                                    \
  do {                                                                      \
    cudaError_t e_ = (call);                                                \
    if (e_ != cudaSuccess) {                                                \
      fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));           \
      return 2;                                                             \
    }                                                                       \
  } while (0)

int main(void) {
  /* x: 1.5 -1.5 0.375 0.0625 0.1875 -0.3125 0.4375 0.625 0.875 1.25 -0.0 1.3125
   *    0.125 -0.03125 0.09375 0.6875 1.0 -1.125 0.25 0.296875, then +0.0 */
  const uint16_t x[32] = {0x3FC0, 0xBFC0, 0x3EC0, 0x3D80, 0x3E40, 0xBEA0, 0x3EE0, 0x3F20,
                          0x3F60, 0x3FA0, 0x8000, 0x3FA8, 0x3E00, 0xBD00, 0x3DC0, 0x3F30,
                          0x3F80, 0xBF90, 0x3E80, 0x3E98};
  const uint8_t want_codes[16] = {0xF7, 0x03, 0xA2, 0x44, 0x66, 0x78, 0x81, 0x51,
                                  0xE6, 0x22, 0, 0, 0, 0, 0, 0};
  const size_t sbytes = mxfp4_scale_bytes(1, 32);
  if (sbytes != 512) {
    fprintf(stderr, "scale bytes %zu\n", sbytes);
    return 1;
  }
  void* dx = NULL;
  uint8_t* dc = NULL;
  uint8_t* ds = NULL;
  void* dy = NULL;
  CHECK_CUDA(cudaMalloc(&dx, sizeof x));
  CHECK_CUDA(cudaMalloc((void**)&dc, 16));
  CHECK_CUDA(cudaMalloc((void**)&ds, sbytes));
  CHECK_CUDA(cudaMalloc(&dy, sizeof x));
  CHECK_CUDA(cudaMemcpy(dx, x, sizeof x, cudaMemcpyHostToDevice));
  int rc = mxfp4_quantize(dx, 1, 32, 32, dc, ds, NULL);
  if (rc != MXFP4_OK) {
    fprintf(stderr, "mxfp4_quantize: %s\n", mxfp4_status_string(rc));
    return 1;
  }
  rc = mxfp4_dequantize(dc, ds, 1, 32, dy, NULL);
  if (rc != MXFP4_OK) {
    fprintf(stderr, "mxfp4_dequantize: %s\n", mxfp4_status_string(rc));
    return 1;
  }
  uint8_t codes[16], scales[512];
  uint16_t y[32];
  CHECK_CUDA(cudaMemcpy(codes, dc, 16, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(scales, ds, sbytes, cudaMemcpyDeviceToHost));
  CHECK_CUDA(cudaMemcpy(y, dy, sizeof y, cudaMemcpyDeviceToHost));
  if (memcmp(codes, want_codes, 16) != 0) {
    fprintf(stderr, "codes differ\n");
    return 1;
  }
  for (size_t i = 0; i < sbytes; ++i) {
    if (scales[i] != (i == 0 ? 125 : 0)) {
      fprintf(stderr, "scale byte %zu = %u\n", i, scales[i]);
      return 1;
    }
  }
  /* dequantized: code * 2^-2 -> 1.5 -1.5 0.375 0 0.25 -0.25 0.5 0.5 1 1 -0 1.5 ... */
  const uint16_t want_y[12] = {0x3FC0, 0xBFC0, 0x3EC0, 0x0000, 0x3E80, 0xBE80,
                               0x3F00, 0x3F00, 0x3F80, 0x3F80, 0x8000, 0x3FC0};
  if (memcmp(y, want_y, sizeof want_y) != 0) {
    fprintf(stderr, "dequantized values differ\n");
    return 1;
  }
  /* host-side validation: K not a multiple of 32 */
  if (mxfp4_quantize(dx, 1, 33, 33, dc, ds, NULL) != MXFP4_ESHAPE) return 1;
  cudaFree(dx);
  cudaFree(dc);
  cudaFree(ds);
  cudaFree(dy);
  printf("c abi: quantize + dequantize of the worked block match\n");
  return 0;
}
