// quantize.cu — BF16 -> MXFP4 (E2M1 codes + 128x4-tiled E8M0 scales), dense
// and per-expert grouped, for sm_103a.
//
// Method: vLLM PR #43557 page ("Fix the E8M0 scale computation in the MXFP4
// MoE CUTLASS kernel"), "Implementation breakdown" items 1 and 3, the
// cvt_warp_fp16_to_fp4 excerpt (UE8M0 branch) and the untile_cutlass_scale
// snippet (tiled layout).  Element rounding: OCP MX E2M1, round to nearest
// even, saturating at +-6; blocks whose scale exponent is 0 emit zero codes.
//
// Work decomposition.  One CTA (256 threads) owns one 128-row x 128-column
// tile: exactly the rows and scale columns of one 512-byte chunk of the tiled
// scale layout, so the chunk is assembled in shared memory and leaves the SM
// as 32 coalesced 16-byte stores.  Lane l of a warp covers 8 BF16 elements
// (one 16-byte load) of row (2*warp + l/16) of a 16-row pass; four lanes form
// one 32-element block, reduced with two xor-shuffles.  All eight passes'
// loads are issued before any compute (32 KB in flight per CTA).
// Each 16-lane half-warp writes 64 contiguous code bytes per row.
#include <cuda_runtime.h>

#include "mxfp4_device.cuh"
#include "mxfp4_internal.h"
#include "../../include/mxfp4.h"

namespace mxfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kPasses = kTileRows / (2 * (kThreads / 32));  // 8 passes of 16 rows

struct QuantizeParams {
  const uint8_t* __restrict__ x;  // BF16 bytes
  int64_t ldx_bytes;              // input row stride in bytes
  int64_t M;                      // rows (dense only)
  int64_t code_ld;                // bytes per code row = K/2
  uint8_t* __restrict__ codes;
  uint8_t* __restrict__ scales;
  int32_t sK;                     // scale columns K/32
  int32_t nKT;                    // k tiles ceil(sK/4)
  const int32_t* __restrict__ offsets;  // grouped: input row offsets [E+1]
  const int32_t* __restrict__ padded;   // grouped: padded row offsets [E+1]
  int32_t E;
};

// Segment holding padded row `prow`: the last e in [0, E) with P[e] <= prow
// (empty segments share their start with the next one, so the last such e
// is never empty when prow < P[E]).
__device__ __forceinline__ int find_segment(const int32_t* __restrict__ P, int E, int64_t prow) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(__ldg(P + mid)) <= prow) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <bool kGrouped>
__global__ void __launch_bounds__(kThreads) quantize_tiles_kernel(const QuantizeParams p) {
  const int kt = static_cast<int>(blockIdx.x % static_cast<uint32_t>(p.nKT));
  const int64_t tile = blockIdx.x / static_cast<uint32_t>(p.nKT);

  int64_t row0, row_end;
  if constexpr (kGrouped) {
    const int64_t total_padded = __ldg(p.padded + p.E);
    const int64_t prow = tile * kTileRows;
    if (total_padded < 0 || prow >= total_padded) return;  // bad offsets / past the end
    const int e = find_segment(p.padded, p.E, prow);
    row0 = __ldg(p.offsets + e) + (prow - __ldg(p.padded + e));
    row_end = __ldg(p.offsets + e + 1);
  } else {
    row0 = tile * kTileRows;
    row_end = p.M;
  }

  __shared__ __align__(16) uint8_t chunk[kChunkBytes];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int seg = lane & 15;        // 8-element segment inside the 128 columns
  const int blk = seg >> 2;         // scale column inside the tile (0..3)
  const bool col_ok = kt * kTileBlocks + blk < p.sK;
  const int64_t col_byte = static_cast<int64_t>(kt) * (kTileCols * 2) + seg * 16;

  uint4 v[kPasses];
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    const int lr = i * 16 + warp * 2 + (lane >> 4);
    const int64_t r = row0 + lr;
    v[i] = make_uint4(0u, 0u, 0u, 0u);
    if (col_ok && r < row_end) v[i] = ld_stream_v4(p.x + r * p.ldx_bytes + col_byte);
  }

#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    const int lr = i * 16 + warp * 2 + (lane >> 4);
    const int64_t r = row0 + lr;
    // block absmax on BF16 bit patterns: with the sign cleared, the unsigned
    // order of the patterns is the order of the magnitudes.
    const uint32_t m2 = vmax_u16x2(vmax_u16x2(v[i].x & 0x7FFF7FFFu, v[i].y & 0x7FFF7FFFu),
                                   vmax_u16x2(v[i].z & 0x7FFF7FFFu, v[i].w & 0x7FFF7FFFu));
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    const uint32_t s = e8m0_from_absmax_bf16(m);
    if ((lane & 3) == 0) chunk[chunk_offset(lr, blk)] = static_cast<uint8_t>(s);

    // x * 2^(127-s): exact power-of-two scaling of BF16 values in float32.
    const float inv = inv_scale_from_e8m0(s);
    uint32_t code = cvt_e2m1x8(__uint_as_float(v[i].x << 16) * inv,
                               __uint_as_float(v[i].x & 0xFFFF0000u) * inv,
                               __uint_as_float(v[i].y << 16) * inv,
                               __uint_as_float(v[i].y & 0xFFFF0000u) * inv,
                               __uint_as_float(v[i].z << 16) * inv,
                               __uint_as_float(v[i].z & 0xFFFF0000u) * inv,
                               __uint_as_float(v[i].w << 16) * inv,
                               __uint_as_float(v[i].w & 0xFFFF0000u) * inv);
    if (s == 0u) code = 0u;
    if (col_ok && r < row_end)
      st_stream_u32(p.codes + r * p.code_ld + static_cast<int64_t>(kt) * (kTileCols / 2) + seg * 4,
                    code);
  }

  __syncthreads();
  if (threadIdx.x < kChunkBytes / 16) {
    const int64_t c = tile * p.nKT + kt;
    const uint4 w = reinterpret_cast<const uint4*>(chunk)[threadIdx.x];
    st_stream_v4(p.scales + c * kChunkBytes + threadIdx.x * 16, w);
  }
}

// Validates 0 = o[0] <= o[1] <= ... <= o[E] = total_rows and writes the
// padded row starts P[e] = sum_{e'<e} ceil(n_e'/128)*128 (P[E] = total).
// One CTA of 1024 threads; a block-wide scan per 1024 segments.
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads)
grouped_offsets_kernel(const int32_t* __restrict__ off, int32_t E, int64_t total_rows,
                       int32_t* __restrict__ padded, int32_t* __restrict__ status) {
  __shared__ int s_bad;
  __shared__ int64_t s_warp[kScanThreads / 32];
  __shared__ int64_t s_carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_bad = (off[0] != 0) || (static_cast<int64_t>(off[E]) != total_rows);
    s_carry = 0;
  }
  __syncthreads();
  for (int base = 0; base < E; base += kScanThreads) {
    const int e = base + tid;
    int64_t cnt = 0;
    if (e < E) {
      const int64_t a = off[e], b = off[e + 1];
      if (b < a) atomicOr(&s_bad, 1);
      else cnt = (b - a + kTileRows - 1) / kTileRows * kTileRows;
    }
    int64_t inc = cnt;  // inclusive warp scan
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t t = __shfl_up_sync(0xFFFFFFFFu, inc, d);
      if (lane >= d) inc += t;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      int64_t w = s_warp[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int64_t t = __shfl_up_sync(0xFFFFFFFFu, w, d);
        if (lane >= d) w += t;
      }
      s_warp[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int64_t before = s_carry + (warp > 0 ? s_warp[warp - 1] : 0) + inc - cnt;
    if (e < E) padded[e] = static_cast<int32_t>(before);
    __syncthreads();
    if (tid == 0) s_carry += s_warp[kScanThreads / 32 - 1];
    __syncthreads();
  }
  if (tid == 0) padded[E] = static_cast<int32_t>(s_carry);
  __syncthreads();
  if (s_bad) {
    for (int e = tid; e <= E; e += kScanThreads) padded[e] = -1;
  }
  if (tid == 0 && status != nullptr) *status = s_bad ? MXFP4_EOFFSETS : MXFP4_OK;
}

}  // namespace

cudaError_t launch_quantize(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes,
                            uint8_t* scales, cudaStream_t stream) {
  QuantizeParams p{};
  p.x = static_cast<const uint8_t*>(x);
  p.ldx_bytes = ldx * 2;
  p.M = M;
  p.code_ld = K / 2;
  p.codes = codes;
  p.scales = scales;
  p.sK = static_cast<int32_t>(K / kBlock);
  p.nKT = (p.sK + kTileBlocks - 1) / kTileBlocks;
  const int64_t tiles = (M + kTileRows - 1) / kTileRows;
  const unsigned grid = static_cast<unsigned>(tiles * p.nKT);
  quantize_tiles_kernel<false><<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_quantize_grouped(const void* x, int64_t total_rows, int64_t K,
                                    const int32_t* offsets, int32_t E, uint8_t* codes,
                                    uint8_t* scales, int32_t* scale_row_offsets,
                                    int32_t* status, int64_t bound_tiles, cudaStream_t stream) {
  grouped_offsets_kernel<<<1, kScanThreads, 0, stream>>>(offsets, E, total_rows,
                                                         scale_row_offsets, status);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess || E == 0 || bound_tiles == 0) return err;
  QuantizeParams p{};
  p.x = static_cast<const uint8_t*>(x);
  p.ldx_bytes = K * 2;
  p.M = total_rows;
  p.code_ld = K / 2;
  p.codes = codes;
  p.scales = scales;
  p.sK = static_cast<int32_t>(K / kBlock);
  p.nKT = (p.sK + kTileBlocks - 1) / kTileBlocks;
  p.offsets = offsets;
  p.padded = scale_row_offsets;
  p.E = E;
  const unsigned grid = static_cast<unsigned>(bound_tiles * p.nKT);
  quantize_tiles_kernel<true><<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mxfp4
