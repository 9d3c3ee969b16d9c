// dequantize.cu — MXFP4 (packed E2M1 codes + 128x4-tiled E8M0 scales) -> BF16
// for sm_103a.
//
// Method: the inverse of the format.  vLLM PR #46915 page ("Fix the SM90
// MXFP4 MoE test weight/scale interleave"), "Motivation": packed FP4 weights
// are read back through an FP4 -> BF16 table, so the scale byte of each
// element must be found at the right place of the interleaved layout; PR
// #43557 page, cvt_warp_fp16_to_fp4 excerpt: the scale value is 2^(s-127)
// built from the exponent bits; untile_cutlass_scale: the tiled layout.
//   y = BF16_RNE(e2m1(code) * 2^(s-127)); s == 255 (E8M0 NaN) -> 0x7FC0.
// The product has at most two significant bits, so the only rounding is
// overflow to +-Inf (s >= 253) — no double rounding through float32.
//
// Same tiles as the quantizer: one CTA per 128x128 tile (one 512-byte scale
// chunk).  Lane l of warp w handles 8 elements of row 2*w + l/16 in each of
// 8 passes of 16 rows: a 4-byte code load, one scale byte of the chunk and a
// 16-byte BF16 store, so each warp store instruction writes two full 256-byte
// row segments.  All loads of a CTA are issued before any compute.  Launched
// with programmatic dependent launch.
#include <cuda_runtime.h>

#include "mxfp4_device.cuh"
#include "mxfp4_internal.h"

namespace mxfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kPasses = kTileRows / (2 * (kThreads / 32));  // 8 passes of 16 rows

struct DequantizeParams {
  const uint8_t* __restrict__ codes;
  const uint8_t* __restrict__ scales;
  uint8_t* __restrict__ y;  // BF16 bytes
  int64_t M;
  int64_t code_ld;  // K/2 bytes
  int64_t y_ld;     // 2K bytes
  int32_t sK;
  int32_t nKT;
};

// Four code bytes (8 elements, element 2j in the low nibble of byte j) and a
// scale value -> 16 bytes of BF16.
__device__ __forceinline__ uint4 decode8(uint32_t c, float sc) {
  uint4 o;
  uint32_t h;
  h = cvt_e2m1x2_to_f16x2(c);
  o.x = cvt_bf16x2(half_lo_to_f32(h) * sc, half_hi_to_f32(h) * sc);
  h = cvt_e2m1x2_to_f16x2(c >> 8);
  o.y = cvt_bf16x2(half_lo_to_f32(h) * sc, half_hi_to_f32(h) * sc);
  h = cvt_e2m1x2_to_f16x2(c >> 16);
  o.z = cvt_bf16x2(half_lo_to_f32(h) * sc, half_hi_to_f32(h) * sc);
  h = cvt_e2m1x2_to_f16x2(c >> 24);
  o.w = cvt_bf16x2(half_lo_to_f32(h) * sc, half_hi_to_f32(h) * sc);
  return o;
}

__global__ void __launch_bounds__(kThreads) dequantize_tiles_kernel(const DequantizeParams p) {
  pdl_wait();
  pdl_release();
  const int kt = static_cast<int>(blockIdx.x % static_cast<uint32_t>(p.nKT));
  const int64_t tile = blockIdx.x / static_cast<uint32_t>(p.nKT);
  const int64_t row0 = tile * kTileRows;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int seg = lane & 15;  // 8-element segment inside the 128 columns
  const int blk = seg >> 2;   // scale column inside the tile
  const bool col_ok = kt * kTileBlocks + blk < p.sK;
  const uint8_t* chunk = p.scales + (tile * p.nKT + kt) * kChunkBytes;

  uint32_t c[kPasses];
  uint32_t s[kPasses];
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    const int lr = i * 16 + warp * 2 + (lane >> 4);
    const int64_t r = row0 + lr;
    c[i] = 0u;
    s[i] = 0u;
    if (col_ok && r < p.M) {
      c[i] = ld_stream_u32(p.codes + r * p.code_ld + static_cast<int64_t>(kt) * (kTileCols / 2) +
                           seg * 4);
      s[i] = __ldg(chunk + chunk_offset(lr, blk));
    }
  }
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    const int lr = i * 16 + warp * 2 + (lane >> 4);
    const int64_t r = row0 + lr;
    uint4 o;
    if (s[i] == 255u) {
      o = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
    } else {
      o = decode8(c[i], scale_from_e8m0(s[i]));
    }
    if (col_ok && r < p.M)
      st_stream_v4(p.y + r * p.y_ld + static_cast<int64_t>(kt) * (kTileCols * 2) + seg * 16, o);
  }
}

}  // namespace

cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t M, int64_t K,
                              void* y, cudaStream_t stream) {
  DequantizeParams p{};
  p.codes = codes;
  p.scales = scales;
  p.y = static_cast<uint8_t*>(y);
  p.M = M;
  p.code_ld = K / 2;
  p.y_ld = K * 2;
  p.sK = static_cast<int32_t>(K / kBlock);
  p.nKT = (p.sK + kTileBlocks - 1) / kTileBlocks;
  const int64_t tiles = (M + kTileRows - 1) / kTileRows;
  return launch_pdl(dequantize_tiles_kernel, static_cast<unsigned>(tiles * p.nKT), kThreads, 0,
                    stream, p);
}

}  // namespace mxfp4
