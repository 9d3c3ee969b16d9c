// swap_w13.cu — fused gate/up weights [w1; w3] -> [w3; w1] for MXFP4 codes,
// E8M0 scales (flat or 128x4-tiled per expert) and the biases, on sm_103a.
//
// Method: vLLM PR #51038 page ("[Bugfix][Quantization] Fix MXFP4 conversion
// for FlashInfer CUTLASS"), "Implementation breakdown" item 2 and the
// convert_weight_to_mxfp4_moe_kernel_format branch: per expert, output row r
// of the 2N fused rows is input row (r + N) mod 2N, for codes and scales;
// the w13 bias halves change places and are cast FP32 -> BF16 (RNE); the w2
// bias is cast only.  Tiled scales are swapped by logical row (each output
// 4-byte word of a chunk is one row's 4 scale columns, gathered from the
// source row's word), pad rows and pad columns written as zero.
//
// One launch covers all three parts: the grid is split into a code range
// (one warp per row, 16-byte vector copies), a scale range and a bias range.
#include <algorithm>

#include <cuda_runtime.h>

#include "mxfp4_device.cuh"
#include "mxfp4_internal.h"

namespace mxfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct SwapParams {
  const uint4* __restrict__ codes_in;
  uint4* __restrict__ codes_out;
  int64_t rows;       // E * 2N
  int64_t two_n;
  int64_t half;       // N
  int32_t row_vecs;   // 16-byte vectors per code row = K/32
  // scales
  const uint8_t* __restrict__ scales_in;
  uint8_t* __restrict__ scales_out;
  int32_t tiled;
  int32_t sK;
  int32_t nKT;
  int64_t chunk_words;  // tiled: 4-byte words per expert buffer
  int64_t scale_items;  // tiled: E * chunk_words; flat: E * 2N * sK bytes
  // biases
  const float* __restrict__ b13_in;
  uint16_t* __restrict__ b13_out;
  int64_t b13_numel;    // E * 2N (0 when absent)
  const float* __restrict__ b2_in;
  uint16_t* __restrict__ b2_out;
  int64_t b2_numel;
  // grid split
  uint32_t code_blocks;
  uint32_t scale_blocks;
};

__device__ __forceinline__ int64_t partner_row(int64_t r, int64_t half) {
  return r < half ? r + half : r - half;
}

__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  return static_cast<uint16_t>(cvt_bf16x2(f, 0.0f) & 0xFFFFu);
}

__global__ void __launch_bounds__(kThreads) swap_w13_kernel(const SwapParams p) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  if (blockIdx.x < p.code_blocks) {
    // ---- codes: one warp per row, 16-byte vectors, two rows in flight
    const int64_t stride = static_cast<int64_t>(p.code_blocks) * kWarps;
    for (int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + warp; row < p.rows;
         row += stride) {
      const int64_t e = row / p.two_n;
      const int64_t r = row - e * p.two_n;
      const int64_t src = e * p.two_n + partner_row(r, p.half);
      const uint4* in = p.codes_in + src * p.row_vecs;
      uint4* out = p.codes_out + row * p.row_vecs;
      int v = lane;
      for (; v + 96 < p.row_vecs; v += 128) {
        const uint4 a = ld_stream_v4(in + v), b = ld_stream_v4(in + v + 32);
        const uint4 c = ld_stream_v4(in + v + 64), d = ld_stream_v4(in + v + 96);
        st_stream_v4(out + v, a);
        st_stream_v4(out + v + 32, b);
        st_stream_v4(out + v + 64, c);
        st_stream_v4(out + v + 96, d);
      }
      for (; v < p.row_vecs; v += 32) st_stream_v4(out + v, ld_stream_v4(in + v));
    }
    return;
  }
  const uint32_t bid = blockIdx.x - p.code_blocks;
  if (bid < p.scale_blocks) {
    // ---- scales
    const int64_t stride = static_cast<int64_t>(p.scale_blocks) * kThreads;
    for (int64_t i = static_cast<int64_t>(bid) * kThreads + threadIdx.x; i < p.scale_items;
         i += stride) {
      if (p.tiled) {
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
          val = __ldg(reinterpret_cast<const uint32_t*>(p.scales_in) + src);
          const int valid = p.sK - kt * kTileBlocks;  // real scale columns in this k-tile
          if (valid < 4) val &= (1u << (8 * valid)) - 1u;
        }
        reinterpret_cast<uint32_t*>(p.scales_out)[i] = val;
      } else {
        const int64_t row = i / p.sK;
        const int64_t c = i - row * p.sK;
        const int64_t e = row / p.two_n;
        const int64_t r = row - e * p.two_n;
        p.scales_out[i] = __ldg(p.scales_in + (e * p.two_n + partner_row(r, p.half)) * p.sK + c);
      }
    }
    return;
  }
  // ---- biases (FP32 -> BF16, round to nearest even)
  const uint32_t bb = bid - p.scale_blocks;
  const int64_t stride = static_cast<int64_t>(gridDim.x - p.code_blocks - p.scale_blocks) * kThreads;
  for (int64_t i = static_cast<int64_t>(bb) * kThreads + threadIdx.x; i < p.b13_numel + p.b2_numel;
       i += stride) {
    if (i < p.b13_numel) {
      const int64_t e = i / p.two_n;
      const int64_t j = i - e * p.two_n;
      p.b13_out[i] = f32_to_bf16(__ldg(p.b13_in + e * p.two_n + partner_row(j, p.half)));
    } else {
      const int64_t k = i - p.b13_numel;
      p.b2_out[k] = f32_to_bf16(__ldg(p.b2_in + k));
    }
  }
}

}  // namespace

cudaError_t launch_swap_w13(const SwapArgs& a, cudaStream_t stream) {
  SwapParams p{};
  p.codes_in = reinterpret_cast<const uint4*>(a.codes_in);
  p.codes_out = reinterpret_cast<uint4*>(a.codes_out);
  p.rows = static_cast<int64_t>(a.E) * a.two_n;
  p.two_n = a.two_n;
  p.half = a.two_n / 2;
  p.row_vecs = static_cast<int32_t>(a.K / 32);
  p.scales_in = a.scales_in;
  p.scales_out = a.scales_out;
  p.tiled = a.scales_tiled;
  p.sK = static_cast<int32_t>(a.K / kBlock);
  p.nKT = (p.sK + kTileBlocks - 1) / kTileBlocks;
  if (a.scales_tiled) {
    const int64_t tiles = (a.two_n + kTileRows - 1) / kTileRows;
    p.chunk_words = tiles * p.nKT * (kChunkBytes / 4);
    p.scale_items = static_cast<int64_t>(a.E) * p.chunk_words;
  } else {
    p.chunk_words = 0;
    p.scale_items = static_cast<int64_t>(a.E) * a.two_n * p.sK;
  }
  p.b13_in = a.w13_bias_in;
  p.b13_out = static_cast<uint16_t*>(a.w13_bias_out);
  p.b13_numel = a.w13_bias_in ? static_cast<int64_t>(a.E) * a.two_n : 0;
  p.b2_in = a.w2_bias_in;
  p.b2_out = static_cast<uint16_t*>(a.w2_bias_out);
  p.b2_numel = a.w2_bias_in ? a.w2_bias_numel : 0;

  // Code rows: one warp each, enough CTAs to fill every SM several times over.
  const int64_t sms = sm_count();
  const int64_t cap = sms * 16;
  const int64_t code_blocks = std::min<int64_t>((p.rows + kWarps - 1) / kWarps, cap);
  const int64_t scale_blocks = std::min<int64_t>((p.scale_items + kThreads - 1) / kThreads, sms * 4);
  const int64_t bias_items = p.b13_numel + p.b2_numel;
  const int64_t bias_blocks = std::min<int64_t>((bias_items + kThreads - 1) / kThreads, sms * 2);
  p.code_blocks = static_cast<uint32_t>(code_blocks);
  p.scale_blocks = static_cast<uint32_t>(scale_blocks);
  const int64_t grid = code_blocks + scale_blocks + bias_blocks;
  if (grid == 0) return cudaSuccess;
  swap_w13_kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mxfp4
