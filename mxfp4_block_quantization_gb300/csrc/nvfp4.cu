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
// against 13.33 us at 4 CTAs per SM on a 4096 x 7168 activation).  The block
// steps are in nvfp4_device.cuh; the experts quant with the dispatch fused in
// is in dispatch.cu.
#include <cstdint>

#include <cuda_runtime.h>

#include "mxfp4_device.cuh"
#include "mxfp4_internal.h"
#include "nvfp4_device.cuh"

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

template <bool kVec32, bool kF16>
__global__ void __launch_bounds__(kThreads, 5) nvfp4_quantize_kernel(const Nvfp4Params p) {
  __shared__ __align__(16) uint8_t chunk[2][kChunkBytes];
  const int ct = static_cast<int>(blockIdx.x % static_cast<uint32_t>(p.nCT));
  const int64_t mt = blockIdx.x / static_cast<uint32_t>(p.nCT);
  const int64_t row0 = mt * kTileRows;
  {
    // before the grid-dependency wait: thread t asks the L2 for half t % 2
    // (four blocks, 128 bytes) of tile row t / 2 when that half holds a block
    const int64_t pr = row0 + (threadIdx.x >> 1);
    const int h = threadIdx.x & 1;
    const uint8_t* pp = p.x + pr * p.ldx_bytes + static_cast<int64_t>(ct) * (kCtaCols * 2) + h * 128;
    if (pr < p.M && ct * 8 + 4 * h < p.sK && MXFP4_IN_BOUNDS(p, kDbgXY, pp, 1)) prefetch_l2(pp);
  }
  pdl_wait();
  pdl_release();
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
  const int ct = static_cast<int>(blockIdx.x % static_cast<uint32_t>(p.nCT));
  const int64_t mt = blockIdx.x / static_cast<uint32_t>(p.nCT);
  const int64_t row0 = mt * kTileRows;
  pdl_wait();
  pdl_release();
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
    const uint32_t sb = (word >> (8 * cc)) & 0xFFu;
    uint4 o0, o1;
    if ((sb & 0x7Fu) == 0x7Fu) {  // the E4M3 NaN: the canonical BF16 NaN, as E8M0 255
      o0 = o1 = make_uint4(0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u, 0x7FC07FC0u);
    } else {
      const float sfv = e4m3_to_f32(sb);
      o0 = decode8_nv(c[i].x, sfv, inv_g);
      o1 = decode8_nv(c[i].y, sfv, inv_g);
    }
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
