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
constexpr int kElems = 16;                                  // elements per lane per pass
constexpr int kLanesPerRow = kTileCols / kElems;            // 8
constexpr int kRowsPerPass = (kThreads / 32) * (32 / kLanesPerRow);  // 32
constexpr int kPasses = kTileRows / kRowsPerPass;           // 4

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
  const uint8_t* c;     // code bytes of this thread's pass-0 row
  const uint8_t* s;     // the 16-byte chunk row holding this thread's 4 scale bytes
  uint8_t* y;           // output of this thread's pass-0 row
  int lim;
  bool col_ok;
};

// Lane l of warp w covers elements [16*(l%8), 16*(l%8)+16) of row
// 4*w + l/8 (+32 per pass).  Pass i of that row sits in chunk row
// (4*w + l/8), word i, byte (l%8)/2.
template <bool kPersistent>
__global__ void __launch_bounds__(kThreads) dequantize_tiles_kernel(const DequantizeParams p) {
  pdl_wait();
  pdl_release();
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane & (kLanesPerRow - 1);
  const int blk = sub >> 1;
  const int lr0 = warp * (32 / kLanesPerRow) + (lane >> 3);
  const int64_t cld_pass = p.code_ld * kRowsPerPass;
  const int64_t yld_pass = p.y_ld * kRowsPerPass;

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
          sub * (kElems / 2);
    t.s = p.scales + static_cast<int64_t>(u) * kChunkBytes + lr0 * 16;
    t.y = p.y + (row0 + lr0) * p.y_ld + static_cast<int64_t>(kt) * (kTileCols * 2) +
          sub * (kElems * 2);
    return t;
  };

  Tile cur = make_tile(unit);
  uint2 c[kPasses];
#pragma unroll
  for (int i = 0; i < kPasses; ++i)
    c[i] = (cur.col_ok && kRowsPerPass * i < cur.lim) ? ld_stream_v2(cur.c + i * cld_pass)
                                                      : make_uint2(0u, 0u);
  uint4 srow = ld_stream_v4(cur.s);

  for (;;) {
    int next_unit = 0;
    bool has_next = false;
    Tile nxt = cur;
    const uint4 sr = srow;
    if constexpr (kPersistent) {
      next_unit = unit + static_cast<int>(gridDim.x);
      has_next = next_unit < p.n_units;
      if (has_next) {
        nxt = make_tile(next_unit);
        srow = ld_stream_v4(nxt.s);
      }
    }
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
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
      if (cur.col_ok && kRowsPerPass * i < cur.lim) {
        st_stream_v4(cur.y + i * yld_pass, o0);
        st_stream_v4(cur.y + i * yld_pass + 16, o1);
      }
      if constexpr (kPersistent) {
        if (has_next)
          c[i] = (nxt.col_ok && kRowsPerPass * i < nxt.lim) ? ld_stream_v2(nxt.c + i * cld_pass)
                                                            : make_uint2(0u, 0u);
      }
    }
    if (!has_next) break;
    cur = nxt;
    unit = next_unit;
  }
}

constexpr bool kPersistentDequant = false;

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
  auto kernel = dequantize_tiles_kernel<kPersistentDequant>;
  int64_t grid = p.n_units;
  if (kPersistentDequant) {
    const int64_t resident =
        static_cast<int64_t>(sm_count()) * resident_ctas(kernel, kThreads, 0, g_occ);
    grid = p.n_units < resident ? p.n_units : resident;
  }
  return launch_pdl(kernel, static_cast<unsigned>(grid), kThreads, 0, stream, p);
}

}  // namespace mxfp4
