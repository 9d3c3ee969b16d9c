// nvfp4.cu — NVFP4 variant: BF16 -> E2M1 codes with one FP8 E4M3 scale per
// 16 elements (plus the caller's global scale), and its dequantize, sm_103a.
//
// Method: vLLM PR #43557 page ("Fix the E8M0 scale computation in the MXFP4
// MoE CUTLASS kernel"), "Implementation breakdown" item 1 and the non-UE8M0
// branch of the cvt_warp_fp16_to_fp4 excerpt: block scale =
// SFScaleVal * vecMax / 6 stored as E4M3; "Review highlights": the elements
// are scaled with the E4M3-rounded value (SFValue = float(E4M3 byte)), so
// quantize and dequantize use the same scale.  Readings where the page is
// silent: 16-element blocks, float32 steps each rounded to nearest even
//   q = vecMax / 6; sf = g * q; byte = E4M3(sf); inv = g / float(byte);
//   code = E2M1(x * inv), blocks with byte 0 -> zero codes;
//   dequantize: BF16((e2m1 * float(byte)) * (1 / g)).
// Scales use the same 128x4 tiled layout as MXFP4, on 16-element columns:
// one 512-byte chunk per 128 rows x 64 elements.
//
// Work decomposition: one CTA (256 threads) per 128 rows x 128 columns = two
// scale chunks; lane l of warp w covers one 16-element block of row
// 4*w + l/8 in each of 4 passes of 32 rows, so the block max needs no shuffle.
// Both quantize kernels are bounded to 48 registers, 5 CTAs per SM (12.95 us
// against 13.33 us at 4 CTAs per SM on a 4096 x 7168 activation).
#include <cstdint>

#include <cuda_runtime.h>

#include "mxfp4_device.cuh"
#include "mxfp4_internal.h"
#include "../../include/mxfp4.h"

namespace mxfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kNvBlock = 16;
constexpr int kRowsPerPass = 32;
constexpr int kPasses = kTileRows / kRowsPerPass;  // 4
constexpr int kCtaCols = 128;                       // two 64-column scale chunks

struct Nvfp4Params {
  const uint8_t* __restrict__ x;      // BF16 bytes (quantize)
  uint8_t* __restrict__ codes;
  uint8_t* __restrict__ scales;
  uint8_t* __restrict__ y;            // BF16 bytes (dequantize)
  const float* __restrict__ g;        // device global scale
  int64_t ldx_bytes;
  int64_t M;
  int64_t code_ld;                    // K/2
  int64_t y_ld;                       // 2K
  int32_t sK;                         // 16-element scale columns K/16
  int32_t nKT;                        // chunks per m-tile ceil(sK/4)
  int32_t nCT;                        // CTAs per m-tile ceil(nKT/2)
#ifdef MXFP4_DEBUG_BOUNDS
  DebugRanges dbg;                    // byte ranges of the buffers (bounds build)
#endif
};

enum : int { kDbgXY = 0, kDbgCodes, kDbgScales, kDbgG };

// One lane's 16-element block -> its E4M3 scale byte:
//   q = vecMax / 6; sf = g * q; byte = E4M3(sf).
template <bool kF16>
__device__ __forceinline__ uint32_t nv_scale_byte(const uint4 (&v)[2], float g) {
  uint32_t h;
  if constexpr (kF16) {
    h = max_abs_f16x2(max_abs_f16x2(max_abs_f16x2(v[0].x, v[0].y), max_abs_f16x2(v[0].z, v[0].w)),
                      max_abs_f16x2(max_abs_f16x2(v[1].x, v[1].y), max_abs_f16x2(v[1].z, v[1].w)));
  } else {
    h = max_abs_bf16x2(max_abs_bf16x2(max_abs_bf16x2(v[0].x, v[0].y),
                                      max_abs_bf16x2(v[0].z, v[0].w)),
                       max_abs_bf16x2(max_abs_bf16x2(v[1].x, v[1].y),
                                      max_abs_bf16x2(v[1].z, v[1].w)));
  }
  h &= 0x7FFF7FFFu;
  const uint32_t m = max(h & 0xFFFFu, h >> 16);
  const float vmax = __uint_as_float(kF16 ? f16_bits_to_f32_bits(m) : m << 16);
  const float q = vmax / 6.0f;  // IEEE float32 division (no fast-math)
  return cvt_e4m3_satfinite(g * q);
}

// The block's 8 code bytes: x * inv rounded to E2M1, inv = g / float(byte);
// zero codes for byte 0.
template <bool kF16>
__device__ __forceinline__ uint2 nv_codes(const uint4 (&v)[2], uint32_t byte, float inv) {
  uint2 code = make_uint2(0u, 0u);
  if (byte != 0u) {
    if constexpr (kF16) {
      code.x = scale_cvt_e2m1x8_f16(v[0], inv);
      code.y = scale_cvt_e2m1x8_f16(v[1], inv);
    } else {
      code.x = scale_cvt_e2m1x8(v[0], inv);
      code.y = scale_cvt_e2m1x8(v[1], inv);
    }
  }
  return code;
}

template <bool kVec32, bool kF16>
__global__ void __launch_bounds__(kThreads, 5) nvfp4_quantize_kernel(const Nvfp4Params p) {
  __shared__ __align__(16) uint8_t chunk[2][kChunkBytes];
  pdl_wait();
  pdl_release();
  const int ct = static_cast<int>(blockIdx.x % static_cast<uint32_t>(p.nCT));
  const int64_t mt = blockIdx.x / static_cast<uint32_t>(p.nCT);
  const int64_t row0 = mt * kTileRows;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane & 7;                 // 16-element block inside the 128 columns
  const int half = sub >> 2;                // which of the two chunks
  const int cc = sub & 3;                   // scale column inside the chunk
  const int lr0 = warp * 4 + (lane >> 3);   // row in pass 0 (0..31)
  const int64_t avail = p.M - row0;
  const int lim = static_cast<int>((avail < kTileRows ? avail : kTileRows) - lr0);
  const bool col_ok = ct * 8 + sub < p.sK;
  const uint8_t* xp = p.x + (row0 + lr0) * p.ldx_bytes + static_cast<int64_t>(ct) * (kCtaCols * 2) + sub * 32;
  uint8_t* cp = p.codes + (row0 + lr0) * p.code_ld + static_cast<int64_t>(ct) * (kCtaCols / 2) + sub * 8;
  const int64_t ldx_pass = p.ldx_bytes * kRowsPerPass;
  const int64_t cld_pass = p.code_ld * kRowsPerPass;
  const float g = MXFP4_IN_BOUNDS(p, kDbgG, p.g, 4) ? __ldg(p.g) : 0.0f;

  uint4 v[kPasses][2];
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    v[i][0] = v[i][1] = make_uint4(0u, 0u, 0u, 0u);
    if (col_ok && kRowsPerPass * i < lim && MXFP4_IN_BOUNDS(p, kDbgXY, xp + i * ldx_pass, 32))
      load32<kVec32>(xp + i * ldx_pass, v[i]);
  }
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    const uint32_t byte = nv_scale_byte<kF16>(v[i], g);
    chunk[half][lr0 * 16 + i * 4 + cc] = static_cast<uint8_t>(byte);
    const uint2 code = nv_codes<kF16>(v[i], byte, byte != 0u ? g / e4m3_to_f32(byte) : 0.0f);
    if (col_ok && kRowsPerPass * i < lim && MXFP4_IN_BOUNDS(p, kDbgCodes, cp + i * cld_pass, 8))
      st_stream_v2(cp + i * cld_pass, code);
  }
  __syncthreads();
  if (threadIdx.x < 2 * (kChunkBytes / 16)) {
    const int j = threadIdx.x >> 5;
    const int w = threadIdx.x & 31;
    const int kt = ct * 2 + j;
    uint8_t* const sp = p.scales + (mt * p.nKT + kt) * kChunkBytes + w * 16;
    if (kt < p.nKT && MXFP4_IN_BOUNDS(p, kDbgScales, sp, 16)) {
      const uint4 val = reinterpret_cast<const uint4*>(chunk[j])[w];
      st_stream_v4(sp, val);
    }
  }
}

// NVFP4 experts quant: the same CTA work on the grouped layout.  Segment e
// = rows [o[e], o[e+1]) of a contiguous x, with global scale g[e]; its
// 128-row tiles are the padded tiles [P[e]/128, P[e+1]/128).  A CTA finds its
// segment from its padded tile (as the MXFP4 grouped kernel does), reads only
// the segment's rows and writes its two scale chunks whole (rows past the
// segment end quantize as zeros: the pad).  Its one global scale lets the CTA
// tabulate g / float(byte) for the 128 non-negative E4M3 bytes while its
// loads are in flight (the same IEEE divisions, once per CTA instead of once
// per block); with it the kernel fits 48 registers, 5 CTAs per SM (together
// 429 -> 366 us at the 1.9 GB MoE size).
struct Nvfp4GroupedParams {
  const uint8_t* __restrict__ x;          // BF16 [total_rows, K]
  uint8_t* __restrict__ codes;
  uint8_t* __restrict__ scales;
  const float* __restrict__ g;            // [E] global scales
  const int32_t* __restrict__ offsets;    // [E+1]
  const int32_t* __restrict__ padded;     // [E+1], written by the offsets kernel
  int64_t ldx_bytes;                      // 2K
  int64_t code_ld;                        // K/2
  int32_t sK, nKT, nCT, E;
#ifdef MXFP4_DEBUG_BOUNDS
  DebugRanges dbg;                        // slots: kDbgXY, kDbgCodes, kDbgScales, kDbgG, 4 offsets, 5 padded
#endif
};

template <bool kVec32, bool kF16>
__global__ void __launch_bounds__(kThreads, 5) nvfp4_quantize_grouped_kernel(const Nvfp4GroupedParams p) {
  __shared__ __align__(16) uint8_t chunk[2][kChunkBytes];
  __shared__ float inv_tab[128];  // g[e] / float(byte), byte = 0 .. 127
  pdl_wait();
  pdl_release();
  if (!MXFP4_IN_BOUNDS(p, 5, p.padded, (p.E + 1) * 4) ||
      !MXFP4_IN_BOUNDS(p, 4, p.offsets, (p.E + 1) * 4))
    return;
  const int total_padded = __ldg(p.padded + p.E);
  const int ct = static_cast<int>(blockIdx.x % static_cast<uint32_t>(p.nCT));
  const int64_t mt = blockIdx.x / static_cast<uint32_t>(p.nCT);
  const int prow = static_cast<int>(mt * kTileRows);
  if (total_padded < 0 || prow >= total_padded) return;  // rejected offsets / past the end
  const int e = find_segment(p.padded, p.E, prow, total_padded);
  const int64_t row0 = static_cast<int64_t>(__ldg(p.offsets + e)) + (prow - __ldg(p.padded + e));
  const int64_t row_end = __ldg(p.offsets + e + 1);
  const float g = MXFP4_IN_BOUNDS(p, kDbgG, p.g + e, 4) ? __ldg(p.g + e) : 0.0f;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane & 7;
  const int half = sub >> 2;
  const int cc = sub & 3;
  const int lr0 = warp * 4 + (lane >> 3);
  const int64_t avail = row_end - row0;
  const int lim = static_cast<int>((avail < kTileRows ? avail : kTileRows) - lr0);
  const bool col_ok = ct * 8 + sub < p.sK;
  const uint8_t* xp = p.x + (row0 + lr0) * p.ldx_bytes + static_cast<int64_t>(ct) * (kCtaCols * 2) + sub * 32;
  uint8_t* cp = p.codes + (row0 + lr0) * p.code_ld + static_cast<int64_t>(ct) * (kCtaCols / 2) + sub * 8;
  const int64_t ldx_pass = p.ldx_bytes * kRowsPerPass;
  const int64_t cld_pass = p.code_ld * kRowsPerPass;

  uint4 v[kPasses][2];
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    v[i][0] = v[i][1] = make_uint4(0u, 0u, 0u, 0u);
    if (col_ok && kRowsPerPass * i < lim && MXFP4_IN_BOUNDS(p, kDbgXY, xp + i * ldx_pass, 32))
      load32<kVec32>(xp + i * ldx_pass, v[i]);
  }
  // g / float(byte) for every non-negative E4M3 byte, while the loads land
  if (threadIdx.x < 128) inv_tab[threadIdx.x] = g / e4m3_to_f32(threadIdx.x);
  __syncthreads();
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    const uint32_t byte = nv_scale_byte<kF16>(v[i], g);
    chunk[half][lr0 * 16 + i * 4 + cc] = static_cast<uint8_t>(byte);
    const uint2 code = nv_codes<kF16>(v[i], byte, inv_tab[byte]);
    if (col_ok && kRowsPerPass * i < lim && MXFP4_IN_BOUNDS(p, kDbgCodes, cp + i * cld_pass, 8))
      st_stream_v2(cp + i * cld_pass, code);
  }
  __syncthreads();
  if (threadIdx.x < 2 * (kChunkBytes / 16)) {
    const int j = threadIdx.x >> 5;
    const int w = threadIdx.x & 31;
    const int kt = ct * 2 + j;
    uint8_t* const sp = p.scales + (mt * p.nKT + kt) * kChunkBytes + w * 16;
    if (kt < p.nKT && MXFP4_IN_BOUNDS(p, kDbgScales, sp, 16))
      st_stream_v4(sp, reinterpret_cast<const uint4*>(chunk[j])[w]);
  }
}

// 8 codes (element 2j in the low nibble of byte j) times float(E4M3 scale)
// times 1/g -> 16 bytes of BF16.
__device__ __forceinline__ uint4 decode8_nv(uint32_t c, float sfv, float inv_g) {
  uint4 o;
  uint32_t h;
  h = cvt_e2m1x2_to_f16x2(c);
  o.x = cvt_bf16x2((half_lo_to_f32(h) * sfv) * inv_g, (half_hi_to_f32(h) * sfv) * inv_g);
  h = cvt_e2m1x2_to_f16x2(c >> 8);
  o.y = cvt_bf16x2((half_lo_to_f32(h) * sfv) * inv_g, (half_hi_to_f32(h) * sfv) * inv_g);
  h = cvt_e2m1x2_to_f16x2(c >> 16);
  o.z = cvt_bf16x2((half_lo_to_f32(h) * sfv) * inv_g, (half_hi_to_f32(h) * sfv) * inv_g);
  h = cvt_e2m1x2_to_f16x2(c >> 24);
  o.w = cvt_bf16x2((half_lo_to_f32(h) * sfv) * inv_g, (half_hi_to_f32(h) * sfv) * inv_g);
  return o;
}

template <bool kVec32>
__global__ void __launch_bounds__(kThreads) nvfp4_dequantize_kernel(const Nvfp4Params p) {
  pdl_wait();
  pdl_release();
  const int ct = static_cast<int>(blockIdx.x % static_cast<uint32_t>(p.nCT));
  const int64_t mt = blockIdx.x / static_cast<uint32_t>(p.nCT);
  const int64_t row0 = mt * kTileRows;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane & 7;
  const int half = sub >> 2;
  const int cc = sub & 3;
  const int lr0 = warp * 4 + (lane >> 3);
  const int64_t avail = p.M - row0;
  const int lim = static_cast<int>((avail < kTileRows ? avail : kTileRows) - lr0);
  const bool col_ok = ct * 8 + sub < p.sK;
  const uint8_t* cp = p.codes + (row0 + lr0) * p.code_ld + static_cast<int64_t>(ct) * (kCtaCols / 2) + sub * 8;
  uint8_t* yp = p.y + (row0 + lr0) * p.y_ld + static_cast<int64_t>(ct) * (kCtaCols * 2) + sub * 32;
  const int64_t cld_pass = p.code_ld * kRowsPerPass;
  const int64_t yld_pass = p.y_ld * kRowsPerPass;
  const float inv_g = 1.0f / (MXFP4_IN_BOUNDS(p, kDbgG, p.g, 4) ? __ldg(p.g) : 1.0f);  // IEEE division

  uint2 c[kPasses];
#pragma unroll
  for (int i = 0; i < kPasses; ++i)
    c[i] = (col_ok && kRowsPerPass * i < lim && MXFP4_IN_BOUNDS(p, kDbgCodes, cp + i * cld_pass, 8))
               ? ld_stream_v2(cp + i * cld_pass)
               : make_uint2(0u, 0u);
  uint4 sr = make_uint4(0u, 0u, 0u, 0u);
  const uint8_t* srp = p.scales + (mt * p.nKT + ct * 2 + half) * kChunkBytes + lr0 * 16;
  if (col_ok && MXFP4_IN_BOUNDS(p, kDbgScales, srp, 16)) sr = ld_stream_v4(srp);
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    const uint32_t word = i == 0 ? sr.x : i == 1 ? sr.y : i == 2 ? sr.z : sr.w;
    const float sfv = e4m3_to_f32((word >> (8 * cc)) & 0xFFu);
    const uint4 o0 = decode8_nv(c[i].x, sfv, inv_g);
    const uint4 o1 = decode8_nv(c[i].y, sfv, inv_g);
    if (col_ok && kRowsPerPass * i < lim && MXFP4_IN_BOUNDS(p, kDbgXY, yp + i * yld_pass, 32)) {
      if constexpr (kVec32) {
        st_stream_v8(yp + i * yld_pass, o0, o1);
      } else {
        st_stream_v4(yp + i * yld_pass, o0);
        st_stream_v4(yp + i * yld_pass + 16, o1);
      }
    }
  }
}

Nvfp4Params make_params(int64_t M, int64_t K) {
  Nvfp4Params p{};
  p.M = M;
  p.code_ld = K / 2;
  p.y_ld = K * 2;
  p.sK = static_cast<int32_t>(K / kNvBlock);
  p.nKT = (p.sK + kTileBlocks - 1) / kTileBlocks;
  p.nCT = (p.nKT + 1) / 2;
  return p;
}


// NVFP4 experts quant with the MoE dispatch as a scatter: route j of token t
// lands on row dest_rows[t][j] of the expert-sorted batch, whose segment e
// has global scale g[e].  One warp per token: the row is read once, in passes
// of 512 elements (lane = one 16-element block), and each block's max and
// q = vecMax / 6 are computed once; then, per route, the block's E4M3 byte
// (g[e] * q), inverse scale and codes with that route's global scale (the
// codes of a token differ per expert).  Codes leave as one 256-byte run per
// route and pass; the scale bytes of a k-tile (4 lanes) as one 4-byte word of
// the tiled layout under an L2 evict-last policy, as in the MXFP4 direct
// scatter.  The first E CTAs zero the segments' pad rows.
struct Nvfp4ScatterParams {
  const uint8_t* __restrict__ x;          // 16-bit token rows
  int64_t ldx_bytes;
  int64_t num_tokens;
  const int32_t* __restrict__ dest_rows;  // [num_tokens, top_k], -1 = not dispatched
  const float* __restrict__ g;            // [E] global scales
  uint8_t* __restrict__ codes;
  uint8_t* __restrict__ scales;
  const int32_t* __restrict__ offsets;    // [E+1]
  const int32_t* __restrict__ padded;     // [E+1], written by the offsets kernel
  int32_t* status;                        // may be NULL
  int64_t total_rows;
  int64_t code_ld;                        // K/2
  int32_t top_k;
  int32_t E;
  int32_t sK;                             // K/16
  int32_t nKT;                            // ceil(sK/4)
#ifdef MXFP4_DEBUG_BOUNDS
  DebugRanges dbg;  // kDbgXY: x, kDbgCodes, kDbgScales, kDbgG, 4: offsets, 5: padded,
                    // 6: dest_rows, 7: status
#endif
};

constexpr int kScWarps = kThreads / 32;
constexpr int kScBatch = 4;  // passes with loads in flight together

// Byte offset of the scale word (4 columns of one k-tile) of padded row prow
// in k-tile 0 of the 128x4 tiled layout; k-tile kt adds kt * 512.
__device__ __forceinline__ int64_t nv_word_base(int prow, int nKT) {
  return static_cast<int64_t>(prow >> 7) * nKT * kChunkBytes + (prow & 31) * 16 +
         ((prow & 127) >> 5) * 4;
}

template <bool kF16>
__device__ __forceinline__ float nv_block_q(const uint4 (&v)[2]) {
  uint32_t h;
  if constexpr (kF16) {
    h = max_abs_f16x2(max_abs_f16x2(max_abs_f16x2(v[0].x, v[0].y), max_abs_f16x2(v[0].z, v[0].w)),
                      max_abs_f16x2(max_abs_f16x2(v[1].x, v[1].y), max_abs_f16x2(v[1].z, v[1].w)));
  } else {
    h = max_abs_bf16x2(max_abs_bf16x2(max_abs_bf16x2(v[0].x, v[0].y),
                                      max_abs_bf16x2(v[0].z, v[0].w)),
                       max_abs_bf16x2(max_abs_bf16x2(v[1].x, v[1].y),
                                      max_abs_bf16x2(v[1].z, v[1].w)));
  }
  h &= 0x7FFF7FFFu;
  const uint32_t m = max(h & 0xFFFFu, h >> 16);
  return __uint_as_float(kF16 ? f16_bits_to_f32_bits(m) : m << 16) / 6.0f;  // IEEE division
}

template <bool kVec32, bool kF16>
__global__ void __launch_bounds__(kThreads) nvfp4_scatter_kernel(const Nvfp4ScatterParams p) {
  __shared__ int64_t s_code[kScWarps][MXFP4_SCATTER_MAX_TOP_K];  // d * K/2, or -1
  __shared__ int64_t s_word[kScWarps][MXFP4_SCATTER_MAX_TOP_K];  // scale word base
  __shared__ float s_g[kScWarps][MXFP4_SCATTER_MAX_TOP_K];       // the route's global scale

  pdl_wait();
  pdl_release();

  if (!MXFP4_IN_BOUNDS(p, 5, p.padded, (p.E + 1) * 4) ||
      !MXFP4_IN_BOUNDS(p, 4, p.offsets, (p.E + 1) * 4))
    return;
  if (__ldg(p.padded + p.E) < 0) return;  // rejected offsets: nothing is written

  if (static_cast<int>(blockIdx.x) < p.E) {
    // pad rows [n, ceil128(n)) of segment e: zero scale words, row-fastest
    const int e = blockIdx.x;
    const int n = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
    const int npad = ((n + kTileRows - 1) / kTileRows) * kTileRows - n;
    const int P0 = __ldg(p.padded + e) + n;
    const uint64_t keep = l2_evict_last_policy();
    for (int i = threadIdx.x; i < npad * p.nKT; i += kThreads) {
      const int kt = i / npad;
      uint8_t* wp = p.scales + nv_word_base(P0 + (i - kt * npad), p.nKT) + kt * kChunkBytes;
      if (MXFP4_IN_BOUNDS(p, kDbgScales, wp, 4)) st_keep_u32(wp, 0u, keep);
    }
    return;
  }

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x - p.E) * kScWarps + warp;
  if (t >= p.num_tokens) return;  // whole warp; no block-wide barrier below

  // routes, one per lane
  int64_t co = -1, wo = -1;
  float ge = 0.0f;
  bool bad = false;
  if (lane < p.top_k) {
    const int32_t* dp = p.dest_rows + t * p.top_k + lane;
    const int32_t v = MXFP4_IN_BOUNDS(p, 6, dp, 4) ? __ldg(dp) : -1;
    if (v >= 0 && v < p.total_rows) {
      const int e = find_segment(p.offsets, p.E, v, static_cast<int>(p.total_rows));
      co = static_cast<int64_t>(v) * p.code_ld;
      wo = nv_word_base(__ldg(p.padded + e) + (v - __ldg(p.offsets + e)), p.nKT);
      ge = MXFP4_IN_BOUNDS(p, kDbgG, p.g + e, 4) ? __ldg(p.g + e) : 0.0f;
    } else {
      bad = v != -1;
    }
  }
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && p.status != nullptr &&
      MXFP4_IN_BOUNDS(p, 7, p.status, 4))
    atomicExch(p.status, MXFP4_EINDEX);
  s_code[warp][lane] = co;
  s_word[warp][lane] = wo;
  s_g[warp][lane] = ge;
  __syncwarp();

  const uint8_t* xrow = p.x + t * p.ldx_bytes + lane * 32;
  const int n_pass = (p.sK + 31) / 32;  // 32 blocks per pass
  const uint64_t keep = l2_evict_last_policy();
  for (int p0 = 0; p0 < n_pass; p0 += kScBatch) {
    uint4 v[kScBatch][2];
    float q[kScBatch];
#pragma unroll
    for (int b = 0; b < kScBatch; ++b) {
      v[b][0] = v[b][1] = make_uint4(0u, 0u, 0u, 0u);
      const int blk = (p0 + b) * 32 + lane;
      const uint8_t* xp = xrow + static_cast<int64_t>(p0 + b) * 1024;
      if (p0 + b < n_pass && blk < p.sK && MXFP4_IN_BOUNDS(p, kDbgXY, xp, 32))
        load32<kVec32>(xp, v[b]);
    }
#pragma unroll
    for (int b = 0; b < kScBatch; ++b) q[b] = nv_block_q<kF16>(v[b]);
    for (int j = 0; j < p.top_k; ++j) {
      const int64_t c = s_code[warp][j];
      if (c < 0) continue;  // the same for every lane of the warp
      const int64_t w = s_word[warp][j];
      const float g = s_g[warp][j];
#pragma unroll
      for (int b = 0; b < kScBatch; ++b) {
        const int pass = p0 + b;
        const int blk = pass * 32 + lane;
        const uint32_t byte = cvt_e4m3_satfinite(g * q[b]);
        const uint2 code = nv_codes<kF16>(v[b], byte, byte != 0u ? g / e4m3_to_f32(byte) : 0.0f);
        uint8_t* const cp = p.codes + c + static_cast<int64_t>(blk) * 8;
        if (pass < n_pass && blk < p.sK && MXFP4_IN_BOUNDS(p, kDbgCodes, cp, 8))
          st_stream_v2(cp, code);
        // scale word of k-tile pass*8 + lane/4: the bytes of lanes +0..+3
        const uint32_t word = byte | (__shfl_down_sync(0xFFFFFFFFu, byte, 1) << 8) |
                              (__shfl_down_sync(0xFFFFFFFFu, byte, 2) << 16) |
                              (__shfl_down_sync(0xFFFFFFFFu, byte, 3) << 24);
        const int kt = pass * 8 + (lane >> 2);
        uint8_t* const wp = p.scales + w + static_cast<int64_t>(kt) * kChunkBytes;
        if (pass < n_pass && (lane & 3) == 0 && kt < p.nKT &&
            MXFP4_IN_BOUNDS(p, kDbgScales, wp, 4))
          st_keep_u32(wp, word, keep);
      }
    }
  }
}

}  // namespace

cudaError_t launch_quantize_nvfp4(const void* x, int64_t M, int64_t K, int64_t ldx,
                                  const float* global_scale, uint8_t* codes, uint8_t* scales,
                                  bool f16, cudaStream_t stream) {
  Nvfp4Params p = make_params(M, K);
  p.x = static_cast<const uint8_t*>(x);
  p.ldx_bytes = ldx * 2;
  p.codes = codes;
  p.scales = scales;
  p.g = global_scale;
  const int64_t grid = (M + kTileRows - 1) / kTileRows * p.nCT;
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(p.dbg, kDbgXY, x, ((M - 1) * ldx + K) * 2);
  debug_range(p.dbg, kDbgCodes, codes, M * (K / 2));
  debug_range(p.dbg, kDbgScales, scales, (M + kTileRows - 1) / kTileRows * p.nKT * kChunkBytes);
  debug_range(p.dbg, kDbgG, global_scale, 4);
#endif
  const bool v32 = reinterpret_cast<uintptr_t>(x) % 32 == 0 && p.ldx_bytes % 32 == 0;
  const auto kernel = f16 ? (v32 ? nvfp4_quantize_kernel<true, true>
                                 : nvfp4_quantize_kernel<false, true>)
                          : (v32 ? nvfp4_quantize_kernel<true, false>
                                 : nvfp4_quantize_kernel<false, false>);
  return launch_pdl(kernel, static_cast<unsigned>(grid), kThreads, 0, stream, p);
}

cudaError_t launch_quantize_nvfp4_grouped(const void* x, int64_t total_rows, int64_t K,
                                          const int32_t* offsets, int32_t E,
                                          const float* global_scales, uint8_t* codes,
                                          uint8_t* scales, int32_t* scale_row_offsets,
                                          int32_t* status, int64_t bound_tiles, bool f16,
                                          cudaStream_t stream) {
  cudaError_t err = launch_offsets(offsets, E, total_rows, scale_row_offsets, status, stream);
  if (err != cudaSuccess || E == 0 || bound_tiles == 0) return err;
  const Nvfp4Params d = make_params(total_rows, K);
  Nvfp4GroupedParams p{};
  p.x = static_cast<const uint8_t*>(x);
  p.codes = codes;
  p.scales = scales;
  p.g = global_scales;
  p.offsets = offsets;
  p.padded = scale_row_offsets;
  p.ldx_bytes = K * 2;
  p.code_ld = K / 2;
  p.sK = d.sK;
  p.nKT = d.nKT;
  p.nCT = d.nCT;
  p.E = E;
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(p.dbg, kDbgXY, x, total_rows * K * 2);
  debug_range(p.dbg, kDbgCodes, codes, total_rows * (K / 2));
  debug_range(p.dbg, kDbgScales, scales, bound_tiles * p.nKT * kChunkBytes);
  debug_range(p.dbg, kDbgG, global_scales, static_cast<int64_t>(E) * 4);
  debug_range(p.dbg, 4, offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(p.dbg, 5, scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4);
#endif
  const int64_t grid = bound_tiles * p.nCT;  // CTAs past the real padded total exit at once
  const bool v32 = reinterpret_cast<uintptr_t>(x) % 32 == 0 && p.ldx_bytes % 32 == 0;
  const auto kernel = f16 ? (v32 ? nvfp4_quantize_grouped_kernel<true, true>
                                 : nvfp4_quantize_grouped_kernel<false, true>)
                          : (v32 ? nvfp4_quantize_grouped_kernel<true, false>
                                 : nvfp4_quantize_grouped_kernel<false, false>);
  return launch_pdl(kernel, static_cast<unsigned>(grid), kThreads, 0, stream, p);
}

cudaError_t launch_quantize_nvfp4_grouped_scatter(const void* x, int64_t num_tokens, int64_t K,
                                                  int64_t ldx, const int32_t* dest_rows,
                                                  int32_t top_k, int64_t total_rows,
                                                  const int32_t* offsets, int32_t E,
                                                  const float* global_scales, uint8_t* codes,
                                                  uint8_t* scales, int32_t* scale_row_offsets,
                                                  int32_t* status, int64_t bound_tiles, bool f16,
                                                  cudaStream_t stream) {
  cudaError_t err = launch_offsets(offsets, E, total_rows, scale_row_offsets, status, stream);
  if (err != cudaSuccess || E == 0 || K == 0) return err;
  Nvfp4ScatterParams p{};
  p.x = static_cast<const uint8_t*>(x);
  p.ldx_bytes = ldx * 2;
  p.num_tokens = num_tokens;
  p.dest_rows = dest_rows;
  p.g = global_scales;
  p.codes = codes;
  p.scales = scales;
  p.offsets = offsets;
  p.padded = scale_row_offsets;
  p.status = status;
  p.total_rows = total_rows;
  p.code_ld = K / 2;
  p.top_k = top_k;
  p.E = E;
  p.sK = static_cast<int32_t>(K / kNvBlock);
  p.nKT = (p.sK + kTileBlocks - 1) / kTileBlocks;
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(p.dbg, kDbgXY, x, num_tokens > 0 ? ((num_tokens - 1) * ldx + K) * 2 : 0);
  debug_range(p.dbg, kDbgCodes, codes, total_rows * (K / 2));
  debug_range(p.dbg, kDbgScales, scales, bound_tiles * p.nKT * kChunkBytes);
  debug_range(p.dbg, kDbgG, global_scales, static_cast<int64_t>(E) * 4);
  debug_range(p.dbg, 4, offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(p.dbg, 5, scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(p.dbg, 6, dest_rows, num_tokens * top_k * 4);
  debug_range(p.dbg, 7, status, status ? 4 : 0);
#else
  (void)bound_tiles;
#endif
  const int64_t grid = E + (num_tokens + kScWarps - 1) / kScWarps;
  const bool v32 = vec32_ok(x, p.ldx_bytes);
  const auto kernel = f16 ? (v32 ? nvfp4_scatter_kernel<true, true>
                                 : nvfp4_scatter_kernel<false, true>)
                          : (v32 ? nvfp4_scatter_kernel<true, false>
                                 : nvfp4_scatter_kernel<false, false>);
  return launch_pdl(kernel, static_cast<unsigned>(grid), kThreads, 0, stream, p);
}

cudaError_t launch_dequantize_nvfp4(const uint8_t* codes, const uint8_t* scales,
                                    const float* global_scale, int64_t M, int64_t K, void* y,
                                    cudaStream_t stream) {
  Nvfp4Params p = make_params(M, K);
  p.codes = const_cast<uint8_t*>(codes);
  p.scales = const_cast<uint8_t*>(scales);
  p.y = static_cast<uint8_t*>(y);
  p.g = global_scale;
  const int64_t grid = (M + kTileRows - 1) / kTileRows * p.nCT;
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(p.dbg, kDbgXY, y, M * K * 2);
  debug_range(p.dbg, kDbgCodes, codes, M * (K / 2));
  debug_range(p.dbg, kDbgScales, scales, (M + kTileRows - 1) / kTileRows * p.nKT * kChunkBytes);
  debug_range(p.dbg, kDbgG, global_scale, 4);
#endif
  const bool v32 = reinterpret_cast<uintptr_t>(y) % 32 == 0;  // rows are 2K = 32*(K/16) bytes
  return launch_pdl(v32 ? nvfp4_dequantize_kernel<true> : nvfp4_dequantize_kernel<false>,
                    static_cast<unsigned>(grid), kThreads, 0, stream, p);
}

#ifdef MXFP4_DEBUG_BOUNDS
unsigned int debug_violations_nvfp4() {
  unsigned int v = 0, zero = 0;
  cudaMemcpyFromSymbol(&v, g_debug_violations, sizeof v);
  cudaMemcpyToSymbol(g_debug_violations, &zero, sizeof zero);
  return v;
}
#endif

}  // namespace mxfp4
