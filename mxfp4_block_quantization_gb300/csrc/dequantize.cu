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
// Same tiles as the quantizer (128 rows x 128 columns = one 512-byte scale
// chunk), persistent grid, loads pipelined one tile ahead.  Per tile a thread
// reads 8 code words (one per pass) and the two 16-byte rows of the chunk
// that hold its 8 scale bytes, and writes 8 x 16 bytes of BF16.
#include <cuda_runtime.h>

#include "mxfp4_device.cuh"
#include "mxfp4_internal.h"

namespace mxfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kPasses = kTileRows / (2 * (kThreads / 32));

struct DequantizeParams {
  const uint8_t* __restrict__ codes;
  const uint8_t* __restrict__ scales;
  uint8_t* __restrict__ y;  // BF16 bytes
  int64_t M;
  int64_t code_ld;  // K/2 bytes
  int64_t y_ld;     // 2K bytes
  int32_t sK;
  int32_t nKT;
  int32_t n_units;
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

struct Tile {
  const uint8_t* c;     // code word of this thread's pass-0 row
  const uint8_t* s;     // 16-byte chunk row of pass 0 (pass 1 is +256 bytes)
  uint8_t* y;           // output of this thread's pass-0 row
  int lim;
  bool col_ok;
};

__global__ void __launch_bounds__(kThreads) dequantize_tiles_kernel(const DequantizeParams p) {
  pdl_wait();
  pdl_release();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int seg16 = lane & 15;
  const int blk = seg16 >> 2;
  const int lr0 = warp * 2 + (lane >> 4);  // row in pass 0; passes add 16 rows
  const int64_t cld16 = p.code_ld * 16;
  const int64_t yld16 = p.y_ld * 16;

  int unit = blockIdx.x;
  if (unit >= p.n_units) return;

  auto make_tile = [&](int u) {
    Tile t;
    const int mt = u / p.nKT;
    const int kt = u - mt * p.nKT;
    const int64_t row0 = static_cast<int64_t>(mt) * kTileRows;
    const int64_t avail = p.M - row0;
    t.lim = static_cast<int>((avail < kTileRows ? avail : kTileRows) - lr0);
    t.col_ok = kt * kTileBlocks + blk < p.sK;
    t.c = p.codes + (row0 + lr0) * p.code_ld + static_cast<int64_t>(kt) * (kTileCols / 2) +
          seg16 * 4;
    // pass i sits in chunk row (lr0 + 16*(i&1)) % 32, word (i >> 1)
    t.s = p.scales + static_cast<int64_t>(u) * kChunkBytes + lr0 * 16;
    t.y = p.y + (row0 + lr0) * p.y_ld + static_cast<int64_t>(kt) * (kTileCols * 2) + seg16 * 16;
    return t;
  };

  Tile cur = make_tile(unit);
  uint32_t c[kPasses];
  uint4 srow[2];
#pragma unroll
  for (int i = 0; i < kPasses; ++i) c[i] = (cur.col_ok && 16 * i < cur.lim) ? ld_stream_u32(cur.c + i * cld16) : 0u;
  srow[0] = ld_stream_v4(cur.s);
  srow[1] = ld_stream_v4(cur.s + 256);

  for (;;) {
    const int next_unit = unit + static_cast<int>(gridDim.x);
    const bool has_next = next_unit < p.n_units;
    Tile nxt = cur;
    if (has_next) nxt = make_tile(next_unit);
    const uint4 sr0 = srow[0], sr1 = srow[1];
    if (has_next) {
      srow[0] = ld_stream_v4(nxt.s);
      srow[1] = ld_stream_v4(nxt.s + 256);
    }
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
      const uint4 sr = (i & 1) ? sr1 : sr0;
      const uint32_t word = (i >> 1) == 0 ? sr.x : (i >> 1) == 1 ? sr.y : (i >> 1) == 2 ? sr.z : sr.w;
      const uint32_t s = (word >> (8 * blk)) & 0xFFu;
      uint4 o;
      if (s == 255u) {
        o = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
      } else {
        o = decode8(c[i], scale_from_e8m0(s));
      }
      if (cur.col_ok && 16 * i < cur.lim) st_stream_v4(cur.y + i * yld16, o);
      if (has_next) c[i] = (nxt.col_ok && 16 * i < nxt.lim) ? ld_stream_u32(nxt.c + i * cld16) : 0u;
    }
    if (!has_next) break;
    cur = nxt;
    unit = next_unit;
  }
}

int g_occ[64];

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
  p.n_units = static_cast<int32_t>(tiles * p.nKT);
  const int64_t resident = static_cast<int64_t>(sm_count()) *
                           resident_ctas(dequantize_tiles_kernel, kThreads, 0, g_occ);
  const int64_t grid = p.n_units < resident ? p.n_units : resident;
  return launch_pdl(dequantize_tiles_kernel, static_cast<unsigned>(grid), kThreads, 0, stream, p);
}

}  // namespace mxfp4
