// swap_w13.cu — fused gate/up weights [w1; w3] -> [w3; w1] for MXFP4 codes,
// E8M0 scales (flat or 128x4-tiled per expert) and the biases, on sm_103a.
//
// Method: vLLM PR #51038 page ("[Bugfix][Quantization] Fix MXFP4 conversion
// for FlashInfer CUTLASS"), "Implementation breakdown" item 2 and the
// convert_weight_to_mxfp4_moe_kernel_format branch: per expert, output row r
// of the 2N fused rows is input row (r + N) mod 2N, for codes and scales;
// the w13 bias halves change places and are cast FP32 -> BF16 (RNE); the w2
// bias is cast only.  Tiled scales are swapped by logical row, pad rows and
// pad columns written as zero.
//
// Rows of one expert are contiguous, so for codes the swap is two contiguous
// copies of N*K/2 bytes per expert ("half copies").  The same holds for flat
// scales (N*K/32 bytes) and for tiled scales when N is a multiple of 128
// (whole 128-row tiles).  Otherwise tiled scales are gathered word by word:
// each 4-byte word of a chunk is one row's 4 scale columns.
//
// One launch covers all parts: the grid is split into a code range, a scale
// range and a bias range.  A half-copy CTA moves 32 KB with eight 16-byte
// loads in flight per thread.
#include <algorithm>
#include <climits>

#include <cuda_runtime.h>

#include "mxfp4_device.cuh"
#include "mxfp4_internal.h"

namespace mxfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 8;
constexpr int kVecPerCta = kThreads * kVecPerThread;  // 2048 x 16 B = 32 KB

enum ScaleMode : int32_t { kScaleHalfCopy = 0, kScaleTiledGather = 1, kScaleFlatGather = 2 };

// E experts, each two contiguous halves of `half_vecs` 16-byte vectors;
// out half h of expert e <- in half (1 - h).
struct HalfCopy {
  const uint4* __restrict__ in;
  uint4* __restrict__ out;
  int64_t half_vecs;
  int32_t ctas_per_half;
  int32_t ctas;  // 2 * E * ctas_per_half
};

struct SwapParams {
  HalfCopy codes;
  int32_t scale_mode;
  HalfCopy scales;  // kScaleHalfCopy
  // gather modes
  const uint8_t* __restrict__ scales_in;
  uint8_t* __restrict__ scales_out;
  int64_t two_n;
  int64_t half;       // N
  int32_t sK;
  int32_t nKT;
  int64_t chunk_words;  // tiled: 4-byte words per expert buffer
  int64_t scale_items;  // gather: tiled words or flat bytes
  int32_t scale_ctas;
  // biases
  const float* __restrict__ b13_in;
  uint16_t* __restrict__ b13_out;
  int64_t b13_numel;    // E * 2N (0 when absent)
  const float* __restrict__ b2_in;
  uint16_t* __restrict__ b2_out;
  int64_t b2_numel;
#ifdef MXFP4_DEBUG_BOUNDS
  DebugRanges dbg;      // byte ranges of the eight buffers (bounds build)
#endif
};

enum : int {
  kDbgCodesIn = 0, kDbgCodesOut, kDbgScalesIn, kDbgScalesOut, kDbgB13In, kDbgB13Out, kDbgB2In,
  kDbgB2Out
};

__device__ __forceinline__ int64_t partner_row(int64_t r, int64_t half) {
  return r < half ? r + half : r - half;
}

__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  return static_cast<uint16_t>(cvt_bf16x2(f, 0.0f) & 0xFFFFu);
}

__device__ __forceinline__ void half_copy_cta(const SwapParams& p, const HalfCopy& hc, int b,
                                              int slot_in, int slot_out) {
  const int hi = b / hc.ctas_per_half;
  const int part = b - hi * hc.ctas_per_half;
  const int64_t e = hi >> 1;
  const int h = hi & 1;
  const uint4* src = hc.in + (2 * e + (1 - h)) * hc.half_vecs;
  uint4* dst = hc.out + (2 * e + h) * hc.half_vecs;
  const int64_t base = static_cast<int64_t>(part) * kVecPerCta + threadIdx.x;
  uint4 v[kVecPerThread];
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const int64_t j = base + k * kThreads;
    if (j < hc.half_vecs && MXFP4_IN_BOUNDS(p, slot_in, src + j, 16)) v[k] = ld_stream_v4(src + j);
  }
#pragma unroll
  for (int k = 0; k < kVecPerThread; ++k) {
    const int64_t j = base + k * kThreads;
    if (j < hc.half_vecs && MXFP4_IN_BOUNDS(p, slot_out, dst + j, 16)) st_stream_v4(dst + j, v[k]);
  }
}

__global__ void __launch_bounds__(kThreads) swap_w13_kernel(const SwapParams p) {
  pdl_wait();
  pdl_release();
  int b = static_cast<int>(blockIdx.x);
  if (b < p.codes.ctas) {
    half_copy_cta(p, p.codes, b, kDbgCodesIn, kDbgCodesOut);
    return;
  }
  b -= p.codes.ctas;
  if (b < p.scale_ctas) {
    if (p.scale_mode == kScaleHalfCopy) {
      half_copy_cta(p, p.scales, b, kDbgScalesIn, kDbgScalesOut);
      return;
    }
    const int64_t stride = static_cast<int64_t>(p.scale_ctas) * kThreads;
    for (int64_t i = static_cast<int64_t>(b) * kThreads + threadIdx.x; i < p.scale_items;
         i += stride) {
      if (p.scale_mode == kScaleTiledGather) {
        // word i of the tiled output: expert e, chunk t (= m-tile * nKT + k-tile),
        // word w inside the 512-byte chunk = outerM * 4 + innerM.
        const int64_t e = i / p.chunk_words;
        const int64_t wi = i - e * p.chunk_words;
        const int64_t t = wi >> 7;
        const int w = static_cast<int>(wi & 127);
        const int64_t mt = t / p.nKT;
        const int kt = static_cast<int>(t - mt * p.nKT);
        const int64_t r = mt * kTileRows + (w & 3) * 32 + (w >> 2);
        uint32_t val = 0u;
        if (r < p.two_n) {
          const int64_t q = partner_row(r, p.half);
          const int64_t src = e * p.chunk_words + ((q >> 7) * p.nKT + kt) * 128 + (q & 31) * 4 +
                              ((q & 127) >> 5);
          const uint32_t* sp = reinterpret_cast<const uint32_t*>(p.scales_in) + src;
          val = MXFP4_IN_BOUNDS(p, kDbgScalesIn, sp, 4) ? __ldg(sp) : 0u;
          const int valid = p.sK - kt * kTileBlocks;  // real scale columns in this k-tile
          if (valid < 4) val &= (1u << (8 * valid)) - 1u;
        }
        uint32_t* dp = reinterpret_cast<uint32_t*>(p.scales_out) + i;
        if (MXFP4_IN_BOUNDS(p, kDbgScalesOut, dp, 4)) *dp = val;
      } else {
        const int64_t row = i / p.sK;
        const int64_t c = i - row * p.sK;
        const int64_t e = row / p.two_n;
        const int64_t r = row - e * p.two_n;
        const uint8_t* sp = p.scales_in + (e * p.two_n + partner_row(r, p.half)) * p.sK + c;
        if (MXFP4_IN_BOUNDS(p, kDbgScalesIn, sp, 1) && MXFP4_IN_BOUNDS(p, kDbgScalesOut, p.scales_out + i, 1))
          p.scales_out[i] = __ldg(sp);
      }
    }
    return;
  }
  // ---- biases (FP32 -> BF16, round to nearest even)
  b -= p.scale_ctas;
  const int64_t bias_ctas = static_cast<int64_t>(gridDim.x) - p.codes.ctas - p.scale_ctas;
  const int64_t stride = bias_ctas * kThreads;
  for (int64_t i = static_cast<int64_t>(b) * kThreads + threadIdx.x; i < p.b13_numel + p.b2_numel;
       i += stride) {
    if (i < p.b13_numel) {
      const int64_t e = i / p.two_n;
      const int64_t j = i - e * p.two_n;
      const float* bp = p.b13_in + e * p.two_n + partner_row(j, p.half);
      if (MXFP4_IN_BOUNDS(p, kDbgB13In, bp, 4) && MXFP4_IN_BOUNDS(p, kDbgB13Out, p.b13_out + i, 2))
        p.b13_out[i] = f32_to_bf16(__ldg(bp));
    } else {
      const int64_t k = i - p.b13_numel;
      if (MXFP4_IN_BOUNDS(p, kDbgB2In, p.b2_in + k, 4) && MXFP4_IN_BOUNDS(p, kDbgB2Out, p.b2_out + k, 2))
        p.b2_out[k] = f32_to_bf16(__ldg(p.b2_in + k));
    }
  }
}

HalfCopy make_half_copy(const uint8_t* in, uint8_t* out, int64_t E, int64_t half_bytes,
                        int64_t* ctas) {
  HalfCopy h{};
  h.in = reinterpret_cast<const uint4*>(in);
  h.out = reinterpret_cast<uint4*>(out);
  h.half_vecs = half_bytes / 16;
  const int64_t per = (h.half_vecs + kVecPerCta - 1) / kVecPerCta;
  *ctas = 2 * E * per;
  h.ctas_per_half = static_cast<int32_t>(per < INT_MAX ? per : INT_MAX);
  h.ctas = static_cast<int32_t>(*ctas < INT_MAX ? *ctas : INT_MAX);
  return h;
}

}  // namespace

cudaError_t launch_swap_w13(const SwapArgs& a, cudaStream_t stream) {
  SwapParams p{};
  const int64_t N = a.two_n / 2;
  const int64_t sK = a.K / kBlock;
  p.two_n = a.two_n;
  p.half = N;
  p.sK = static_cast<int32_t>(sK);
  p.nKT = static_cast<int32_t>((sK + kTileBlocks - 1) / kTileBlocks);
  // codes: two contiguous halves of N*K/2 bytes per expert (K/2 is a multiple of 16)
  int64_t code_ctas = 0;
  p.codes = make_half_copy(a.codes_in, a.codes_out, a.E, N * (a.K / 2), &code_ctas);

  const int64_t sms = sm_count();
  int64_t scale_ctas = 0;
  p.scales_in = a.scales_in;
  p.scales_out = a.scales_out;
  if (a.E > 0 && sK > 0) {
    const int64_t flat_half = N * sK;
    if (a.scales_tiled && N % kTileRows == 0) {
      p.scale_mode = kScaleHalfCopy;
      p.scales = make_half_copy(a.scales_in, a.scales_out, a.E,
                                (N / kTileRows) * p.nKT * kChunkBytes, &scale_ctas);
    } else if (!a.scales_tiled && flat_half % 16 == 0) {
      p.scale_mode = kScaleHalfCopy;
      p.scales = make_half_copy(a.scales_in, a.scales_out, a.E, flat_half, &scale_ctas);
    } else if (a.scales_tiled) {
      p.scale_mode = kScaleTiledGather;
      const int64_t tiles = (a.two_n + kTileRows - 1) / kTileRows;
      p.chunk_words = tiles * p.nKT * (kChunkBytes / 4);
      p.scale_items = static_cast<int64_t>(a.E) * p.chunk_words;
      scale_ctas = std::min<int64_t>((p.scale_items + kThreads - 1) / kThreads, sms * 8);
    } else {
      p.scale_mode = kScaleFlatGather;
      p.scale_items = static_cast<int64_t>(a.E) * a.two_n * sK;
      scale_ctas = std::min<int64_t>((p.scale_items + kThreads - 1) / kThreads, sms * 8);
    }
  }
  p.scale_ctas = static_cast<int32_t>(scale_ctas);
  p.b13_in = a.w13_bias_in;
  p.b13_out = static_cast<uint16_t*>(a.w13_bias_out);
  p.b13_numel = a.w13_bias_in ? static_cast<int64_t>(a.E) * a.two_n : 0;
  p.b2_in = a.w2_bias_in;
  p.b2_out = static_cast<uint16_t*>(a.w2_bias_out);
  p.b2_numel = a.w2_bias_in ? a.w2_bias_numel : 0;
  const int64_t bias_items = p.b13_numel + p.b2_numel;
  const int64_t bias_ctas = std::min<int64_t>((bias_items + kThreads - 1) / kThreads, sms * 2);
  const int64_t grid = code_ctas + scale_ctas + bias_ctas;
#ifdef MXFP4_DEBUG_BOUNDS
  {
    const int64_t rows = static_cast<int64_t>(a.E) * a.two_n;
    const int64_t scale_bytes =
        a.scales_tiled ? static_cast<int64_t>(a.E) *
                             ((a.two_n + kTileRows - 1) / kTileRows) * p.nKT * kChunkBytes
                       : rows * sK;
    debug_range(p.dbg, kDbgCodesIn, a.codes_in, rows * (a.K / 2));
    debug_range(p.dbg, kDbgCodesOut, a.codes_out, rows * (a.K / 2));
    debug_range(p.dbg, kDbgScalesIn, a.scales_in, sK > 0 ? scale_bytes : 0);
    debug_range(p.dbg, kDbgScalesOut, a.scales_out, sK > 0 ? scale_bytes : 0);
    debug_range(p.dbg, kDbgB13In, a.w13_bias_in, p.b13_numel * 4);
    debug_range(p.dbg, kDbgB13Out, a.w13_bias_out, p.b13_numel * 2);
    debug_range(p.dbg, kDbgB2In, a.w2_bias_in, p.b2_numel * 4);
    debug_range(p.dbg, kDbgB2Out, a.w2_bias_out, p.b2_numel * 2);
  }
#endif
  if (grid == 0) return cudaSuccess;
  if (grid > INT_MAX / 2) return cudaErrorInvalidConfiguration;
  return launch_pdl(swap_w13_kernel, static_cast<unsigned>(grid), kThreads, 0, stream, p);
}

#ifdef MXFP4_DEBUG_BOUNDS
unsigned int debug_violations_swap() {
  unsigned int v = 0, zero = 0;
  cudaMemcpyFromSymbol(&v, g_debug_violations, sizeof v);
  cudaMemcpyToSymbol(g_debug_violations, &zero, sizeof zero);
  return v;
}
#endif

}  // namespace mxfp4
