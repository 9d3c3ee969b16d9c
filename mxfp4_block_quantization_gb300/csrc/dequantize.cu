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
// Same tiles as the quantizer: one CTA (256 threads) per 128x128 tile (one
// 512-byte scale chunk), all loads issued before any compute, launched with
// programmatic dependent launch.  Two lane mappings:
//  - wide (output 32-byte aligned): lane = 16 elements of one row per pass,
//    4 passes; an 8-byte code load, the tile's 4 scale bytes of the lane from
//    one 16-byte chunk row, one 32-byte store per pass (full sectors);
//  - narrow (output only 16-byte aligned): lane = 8 elements per pass, 8
//    passes; a 4-byte code load, one scale byte, one 16-byte store, so each
//    warp store instruction still writes whole 256-byte row segments.
#include <cstdint>

#include <cuda_runtime.h>

#include "mxfp4_device.cuh"
#include "mxfp4_internal.h"

namespace mxfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kPasses = kTileRows / (2 * (kThreads / 32));  // narrow: 8 passes of 16 rows

struct DequantizeParams {
  const uint8_t* __restrict__ codes;
  const uint8_t* __restrict__ scales;
  uint8_t* __restrict__ y;  // BF16 bytes
  int64_t M;
  int64_t code_ld;  // K/2 bytes
  int64_t y_ld;     // 2K bytes
  int32_t sK;
  int32_t nKT;
#ifdef MXFP4_DEBUG_BOUNDS
  DebugRanges dbg;  // byte ranges of codes, scales, y (bounds build)
#endif
};

enum : int { kDbgCodes = 0, kDbgScales, kDbgY };

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

// Wide mapping: lane l of warp w covers elements [16*(l%8), 16*(l%8)+16) of
// row 4*w + l/8 (+32 per pass); pass i of that row has its scale byte in
// chunk row (4*w + l/8), word i, byte (l%8)/2.
__global__ void __launch_bounds__(kThreads) dequantize_wide_kernel(const DequantizeParams p) {
  constexpr int kRowsPerPass = 32;
  constexpr int kWidePasses = kTileRows / kRowsPerPass;
  pdl_wait();
  pdl_release();
  const int kt = static_cast<int>(blockIdx.x % static_cast<uint32_t>(p.nKT));
  const int64_t tile = blockIdx.x / static_cast<uint32_t>(p.nKT);
  const int64_t row0 = tile * kTileRows;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane & 7;
  const int blk = sub >> 1;
  const int lr0 = warp * 4 + (lane >> 3);
  const int64_t avail = p.M - row0;
  const int lim = static_cast<int>((avail < kTileRows ? avail : kTileRows) - lr0);
  const bool col_ok = kt * kTileBlocks + blk < p.sK;
  const uint8_t* cp = p.codes + (row0 + lr0) * p.code_ld + static_cast<int64_t>(kt) * (kTileCols / 2) + sub * 8;
  uint8_t* yp = p.y + (row0 + lr0) * p.y_ld + static_cast<int64_t>(kt) * (kTileCols * 2) + sub * 32;
  const int64_t cld_pass = p.code_ld * kRowsPerPass;
  const int64_t yld_pass = p.y_ld * kRowsPerPass;

  uint2 c[kWidePasses];
#pragma unroll
  for (int i = 0; i < kWidePasses; ++i)
    c[i] = (col_ok && kRowsPerPass * i < lim && MXFP4_IN_BOUNDS(p, kDbgCodes, cp + i * cld_pass, 8))
               ? ld_stream_v2(cp + i * cld_pass)
               : make_uint2(0u, 0u);
  const uint8_t* srp = p.scales + (tile * p.nKT + kt) * kChunkBytes + lr0 * 16;
  const uint4 sr =
      MXFP4_IN_BOUNDS(p, kDbgScales, srp, 16) ? ld_stream_v4(srp) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int i = 0; i < kWidePasses; ++i) {
    const uint32_t word = i == 0 ? sr.x : i == 1 ? sr.y : i == 2 ? sr.z : sr.w;
    const uint32_t s = (word >> (8 * blk)) & 0xFFu;
    uint4 o0, o1;
    if (s == 255u) {
      o0 = o1 = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
    } else {
      const float sc = scale_from_e8m0(s);
      o0 = decode8(c[i].x, sc);
      o1 = decode8(c[i].y, sc);
    }
    if (col_ok && kRowsPerPass * i < lim && MXFP4_IN_BOUNDS(p, kDbgY, yp + i * yld_pass, 32))
      st_stream_v8(yp + i * yld_pass, o0, o1);
  }
}

// Narrow mapping: lane l of warp w covers 8 elements of row 2*w + l/16 in
// each of 8 passes of 16 rows.
__global__ void __launch_bounds__(kThreads) dequantize_narrow_kernel(const DequantizeParams p) {
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
    const uint8_t* cp = p.codes + r * p.code_ld + static_cast<int64_t>(kt) * (kTileCols / 2) + seg * 4;
    if (col_ok && r < p.M && MXFP4_IN_BOUNDS(p, kDbgCodes, cp, 4) &&
        MXFP4_IN_BOUNDS(p, kDbgScales, chunk + chunk_offset(lr, blk), 1)) {
      c[i] = ld_stream_u32(cp);
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
    uint8_t* yp = p.y + r * p.y_ld + static_cast<int64_t>(kt) * (kTileCols * 2) + seg * 16;
    if (col_ok && r < p.M && MXFP4_IN_BOUNDS(p, kDbgY, yp, 16)) st_stream_v4(yp, o);
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
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(p.dbg, kDbgCodes, codes, M * (K / 2));
  debug_range(p.dbg, kDbgScales, scales, tiles * p.nKT * kChunkBytes);
  debug_range(p.dbg, kDbgY, y, M * K * 2);
#endif
  const bool wide = reinterpret_cast<uintptr_t>(y) % 32 == 0;  // rows are 2K = 64*(K/32) bytes
  return launch_pdl(wide ? dequantize_wide_kernel : dequantize_narrow_kernel,
                    static_cast<unsigned>(tiles * p.nKT), kThreads, 0, stream, p);
}

#ifdef MXFP4_DEBUG_BOUNDS
unsigned int debug_violations_dequantize() {
  unsigned int v = 0, zero = 0;
  cudaMemcpyFromSymbol(&v, g_debug_violations, sizeof v);
  cudaMemcpyToSymbol(g_debug_violations, &zero, sizeof zero);
  return v;
}
#endif

}  // namespace mxfp4
