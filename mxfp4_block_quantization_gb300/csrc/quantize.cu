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
// tile: exactly the rows and scale columns of one 512-byte chunk of the
// tiled scale layout, so the chunk is assembled in shared memory and leaves
// the SM as 32 coalesced 16-byte stores.  Lane l of warp w covers 16 BF16
// elements (one 32-byte load, or two 16-byte loads when the input is only
// 16-byte aligned) of row 4*w + l/8 in each of 4 passes of 32 rows; two lanes
// form one 32-element block, reduced with one xor-shuffle.  All four passes'
// loads are issued before any compute (32 KB in flight per CTA, four to five
// CTAs per SM).  The fused-gather variant (quantize_gather_kernel) keeps one
// 128-row tile per CTA but walks a chunk of k-tiles; the scatter forms, one
// warp per token row, are in dispatch.cu.  Launches use programmatic
// dependent launch, so a grid is already resident when its predecessor in the
// stream drains.
#include <cstdint>

#include <cuda_runtime.h>

#include "mxfp4_device.cuh"
#include "mxfp4_internal.h"
#include "../../include/mxfp4.h"

namespace mxfp4 {
namespace {

constexpr int kThreads = 256;                               // dense and grouped CTAs
constexpr int kGatherThreads = 128;                         // gather CTAs: 8 passes per thread
constexpr int kScanThreads = 1024;                          // single-CTA scans

// Rows covered by one pass of a CTA of `threads` threads (4 rows per warp),
// and passes per 128-row tile.
__host__ __device__ constexpr int rows_per_pass(int threads) { return (threads / 32) * (32 / kLanesPerRow); }
__host__ __device__ constexpr int passes(int threads) { return kTileRows / rows_per_pass(threads); }

struct QuantizeParams {
  const uint8_t* __restrict__ x;  // BF16 bytes
  int64_t ldx_bytes;              // input row stride in bytes
  int64_t M;                      // rows (dense only)
  int64_t code_ld;                // bytes per code row = K/2
  uint8_t* __restrict__ codes;
  uint8_t* __restrict__ scales;
  int32_t sK;                     // scale columns K/32
  int32_t nKT;                    // k tiles ceil(sK/4)
  int32_t n_units;                // dense: tiles * nKT (= grid)
  const int32_t* __restrict__ offsets;  // grouped: input row offsets [E+1]
  const int32_t* __restrict__ padded;   // grouped: padded row offsets [E+1]
  int32_t E;
  const int32_t* __restrict__ row_index;  // gather: source row of every output row
  int64_t num_src_rows;                   // gather: rows of x
  int32_t* status;                        // gather: device status word (may be NULL)
  int32_t n_mtiles;                       // gather: m-tiles of the grid (chunk-major order)
#ifdef MXFP4_DEBUG_BOUNDS
  DebugRanges dbg;                        // byte ranges of the buffers below (bounds build)
#endif
};


// Buffer slots of QuantizeParams::dbg.
enum : int { kDbgX = 0, kDbgCodes, kDbgScales, kDbgOffsets, kDbgPadded, kDbgRowIndex, kDbgStatus };

// Lane l of warp w covers elements [16*(l%8), 16*(l%8)+16) of row
// 4*w + l/8 (+32 per pass): two lanes per 32-element block.
//
// kVec32: every lane's 32 bytes are 32-byte aligned (x and the row stride
// are), so they arrive in one 256-bit load per pass; otherwise two 16-byte
// loads (each then touches half of a 32-byte sector).
//
// kF16: the input is IEEE binary16 instead of BF16 (same method: the block
// max is widened to float32 exactly and the E8M0 rule is applied to its bits).
template <bool kGrouped, bool kVec32, bool kF16 = false>
__global__ void __launch_bounds__(kThreads) quantize_tiles_kernel(const QuantizeParams p) {
  constexpr int kRowsPerPass = rows_per_pass(kThreads);
  constexpr int kPasses = passes(kThreads);
  __shared__ __align__(16) uint8_t chunk[kChunkBytes];

  // Tile order: m-tile-major, so consecutive CTAs read adjacent column slices
  // of the same rows.
  const int unit = blockIdx.x;
  const int mt = unit / p.nKT;
  const int kt = unit - mt * p.nKT;

  if constexpr (!kGrouped) {
    // The dense tile's rows are known before the wait: thread t asks the L2
    // for half t % 2 (two scale blocks, 128 bytes) of tile row t / 2, when
    // that half holds a real block.
    const int64_t pr = static_cast<int64_t>(mt) * kTileRows + (threadIdx.x >> 1);
    const int half = threadIdx.x & 1;
    const uint8_t* pp = p.x + pr * p.ldx_bytes + static_cast<int64_t>(kt) * (kTileCols * 2) +
                        half * (kTileCols);
    if (pr < p.M && kt * kTileBlocks + 2 * half < p.sK && MXFP4_IN_BOUNDS(p, kDbgX, pp, 1))
      prefetch_l2(pp);
  }

  pdl_wait();
  pdl_release();
  int64_t row0, row_end;
  if constexpr (kGrouped) {
    // every offset index read below lies in [0, E]
    if (!MXFP4_IN_BOUNDS(p, kDbgPadded, p.padded, (p.E + 1) * 4) ||
        !MXFP4_IN_BOUNDS(p, kDbgOffsets, p.offsets, (p.E + 1) * 4))
      return;
    const int total_padded = __ldg(p.padded + p.E);
    const int prow = mt * kTileRows;
    if (total_padded < 0 || prow >= total_padded) return;  // rejected offsets / past the end
    const int e = find_segment(p.padded, p.E, prow, total_padded);
    row0 = static_cast<int64_t>(__ldg(p.offsets + e)) + (prow - __ldg(p.padded + e));
    row_end = __ldg(p.offsets + e + 1);
  } else {
    row0 = static_cast<int64_t>(mt) * kTileRows;
    row_end = p.M;
  }

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane & (kLanesPerRow - 1);  // 16-element segment inside the 128 columns
  const int blk = sub >> 1;                   // scale column inside the tile (0..3)
  const int lr0 = warp * (32 / kLanesPerRow) + (lane >> 3);  // row in pass 0
  const int64_t avail = row_end - row0;
  const int lim = static_cast<int>((avail < kTileRows ? avail : kTileRows) - lr0);
  const bool col_ok = kt * kTileBlocks + blk < p.sK;
  const int64_t r = row0 + lr0;
  const uint8_t* xp =
      p.x + r * p.ldx_bytes + static_cast<int64_t>(kt) * (kTileCols * 2) + sub * (kElems * 2);
  uint8_t* cp =
      p.codes + r * p.code_ld + static_cast<int64_t>(kt) * (kTileCols / 2) + sub * (kElems / 2);
  const int64_t ldx_pass = p.ldx_bytes * kRowsPerPass;
  const int64_t cld_pass = p.code_ld * kRowsPerPass;

  uint4 v[kPasses][2];
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    v[i][0] = v[i][1] = make_uint4(0u, 0u, 0u, 0u);
    if (col_ok && kRowsPerPass * i < lim && MXFP4_IN_BOUNDS(p, kDbgX, xp + i * ldx_pass, 32))
      load32<kVec32>(xp + i * ldx_pass, v[i]);
  }

#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    const uint32_t s = lane_block_scale<kF16>(v[i]);
    // rows of pass i sit in chunk row lr0 % 32 (outerM), word (lr0 + rows*i) / 32 (innerM)
    if ((lane & 1) == 0) chunk[chunk_offset(lr0 + kRowsPerPass * i, blk)] = static_cast<uint8_t>(s);
    const uint2 code = lane_codes<kF16>(v[i], s);
    if (col_ok && kRowsPerPass * i < lim && MXFP4_IN_BOUNDS(p, kDbgCodes, cp + i * cld_pass, 8))
      st_stream_v2(cp + i * cld_pass, code);
  }

  __syncthreads();
  // chunk index = m-tile * nKT + k-tile = unit
  uint8_t* const sp = p.scales + static_cast<int64_t>(unit) * kChunkBytes + threadIdx.x * 16;
  if (threadIdx.x < kChunkBytes / 16 && MXFP4_IN_BOUNDS(p, kDbgScales, sp, 16)) {
    const uint4 w = reinterpret_cast<const uint4*>(chunk)[threadIdx.x];
    st_stream_v4(sp, w);
  }
}

// Fused dispatch gather, chunked over K: one CTA (128 threads, 8 passes of 16
// rows) owns one padded 128-row tile and a chunk of kGatherChunkTiles k-tiles
// (1024 columns).  The tile's segment and its 128 source-row indices are
// fetched once; the CTA then walks its k-tiles, each a full 128x128 tile with
// its own 512-byte scale chunk (double-buffered in shared memory, one barrier
// per k-tile).  CTAs are ordered chunk-major, so the resident CTAs read the
// same 1024-column slice of the source rows (32 MB for 16384 rows of 7168),
// which the L2 keeps while the other routes of each row come by.
constexpr int kGatherChunkTiles = 8;

template <bool kVec32, bool kF16>
__global__ void __launch_bounds__(kGatherThreads) quantize_gather_kernel(const QuantizeParams p) {
  constexpr int kRowsPerPass = rows_per_pass(kGatherThreads);
  constexpr int kPasses = passes(kGatherThreads);
  __shared__ __align__(16) uint8_t chunk[2][kChunkBytes];

  pdl_wait();
  pdl_release();

  const int unit = blockIdx.x;
  const int kc = unit / p.n_mtiles;
  const int mt = unit - kc * p.n_mtiles;
  if (!MXFP4_IN_BOUNDS(p, kDbgPadded, p.padded, (p.E + 1) * 4) ||
      !MXFP4_IN_BOUNDS(p, kDbgOffsets, p.offsets, (p.E + 1) * 4))
    return;
  const int total_padded = __ldg(p.padded + p.E);
  const int prow = mt * kTileRows;
  if (total_padded < 0 || prow >= total_padded) return;  // rejected offsets / past the end
  const int e = find_segment(p.padded, p.E, prow, total_padded);
  const int64_t row0 = static_cast<int64_t>(__ldg(p.offsets + e)) + (prow - __ldg(p.padded + e));
  const int64_t row_end = __ldg(p.offsets + e + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane & (kLanesPerRow - 1);
  const int blk = sub >> 1;
  const int lr0 = warp * (32 / kLanesPerRow) + (lane >> 3);
  const int64_t avail = row_end - row0;
  const int lim = static_cast<int>((avail < kTileRows ? avail : kTileRows) - lr0);
  const int64_t r = row0 + lr0;

  // source rows of this thread's eight output rows; an index outside
  // [0, num_src_rows) reads nothing, quantizes as a zero row and is reported
  int64_t src[kPasses];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    src[i] = (kRowsPerPass * i < lim &&
              MXFP4_IN_BOUNDS(p, kDbgRowIndex, p.row_index + r + kRowsPerPass * i, 4))
                 ? __ldg(p.row_index + r + kRowsPerPass * i)
                 : 0;
    const bool in_range = src[i] >= 0 && src[i] < p.num_src_rows;
    if (kRowsPerPass * i < lim) bad |= !in_range;
    src[i] = (kRowsPerPass * i < lim && in_range) ? src[i] : -1;
  }
  if (bad && p.status != nullptr && MXFP4_IN_BOUNDS(p, kDbgStatus, p.status, 4))
    atomicExch(p.status, MXFP4_EINDEX);

  const int kt0 = kc * kGatherChunkTiles;
  const int kt_end = kt0 + kGatherChunkTiles < p.nKT ? kt0 + kGatherChunkTiles : p.nKT;
  const int64_t cld_pass = p.code_ld * kRowsPerPass;
  int buf = 0;
  for (int kt = kt0; kt < kt_end; ++kt) {
    const bool col_ok = kt * kTileBlocks + blk < p.sK;
    const uint8_t* xcol = p.x + static_cast<int64_t>(kt) * (kTileCols * 2) + sub * (kElems * 2);
    uint4 v[kPasses][2];
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
      v[i][0] = v[i][1] = make_uint4(0u, 0u, 0u, 0u);
      if (col_ok && src[i] >= 0 && MXFP4_IN_BOUNDS(p, kDbgX, xcol + src[i] * p.ldx_bytes, 32))
        load32<kVec32>(xcol + src[i] * p.ldx_bytes, v[i]);
    }
    uint8_t* cp = p.codes + r * p.code_ld + static_cast<int64_t>(kt) * (kTileCols / 2) +
                  sub * (kElems / 2);
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
      const uint32_t s = lane_block_scale<kF16>(v[i]);
      if ((lane & 1) == 0)
        chunk[buf][chunk_offset(lr0 + kRowsPerPass * i, blk)] = static_cast<uint8_t>(s);
      const uint2 code = lane_codes<kF16>(v[i], s);
      if (col_ok && kRowsPerPass * i < lim && MXFP4_IN_BOUNDS(p, kDbgCodes, cp + i * cld_pass, 8))
        st_stream_v2(cp + i * cld_pass, code);
    }
    __syncthreads();
    const int64_t c = static_cast<int64_t>(mt) * p.nKT + kt;
    uint8_t* const sp = p.scales + c * kChunkBytes + threadIdx.x * 16;
    if (threadIdx.x < kChunkBytes / 16 && MXFP4_IN_BOUNDS(p, kDbgScales, sp, 16)) {
      const uint4 w = reinterpret_cast<const uint4*>(chunk[buf])[threadIdx.x];
      st_stream_v4(sp, w);
    }
    buf ^= 1;
  }
}

// Validates 0 = o[0] <= o[1] <= ... <= o[E] = total_rows and writes the
// padded row starts P[e] = sum_{e'<e} ceil(n_e'/128)*128 (P[E] = total).
// One CTA of kScanThreads threads; a block-wide scan per kScanThreads segments.

struct OffsetsParams {
  const int32_t* __restrict__ off;
  int32_t E;
  int64_t total_rows;
  int32_t* __restrict__ padded;
  int32_t* __restrict__ status;
#ifdef MXFP4_DEBUG_BOUNDS
  DebugRanges dbg;  // slots kDbgOffsets, kDbgPadded, kDbgStatus
#endif
};

__global__ void __launch_bounds__(kScanThreads) grouped_offsets_kernel(const OffsetsParams q) {
  const int32_t* __restrict__ off = q.off;
  const int32_t E = q.E;
  const int64_t total_rows = q.total_rows;
  int32_t* __restrict__ padded = q.padded;
  int32_t* __restrict__ status = q.status;
  __shared__ int64_t s_warp[kScanThreads / 32];
  pdl_wait();
  pdl_release();
  // every index below lies in [0, E]
  if (!MXFP4_IN_BOUNDS(q, kDbgOffsets, off, (E + 1) * 4) ||
      !MXFP4_IN_BOUNDS(q, kDbgPadded, padded, (E + 1) * 4) ||
      (status != nullptr && !MXFP4_IN_BOUNDS(q, kDbgStatus, status, 4)))
    return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // every thread's loads are in flight at once: the first and last offsets
  // are checked by the threads that load them anyway
  bool bad = E == 0 && (off[0] != 0 || static_cast<int64_t>(off[0]) != total_rows);
  int64_t carry = 0;  // the same in every thread
  for (int base = 0; base < E; base += kScanThreads) {
    const int e = base + tid;
    int64_t cnt = 0;
    if (e < E) {
      const int64_t a = off[e], b = off[e + 1];
      if (b < a || (e == 0 && a != 0) || (e == E - 1 && b != total_rows)) bad = true;
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
    const int64_t before = carry + (warp > 0 ? s_warp[warp - 1] : 0) + inc - cnt;
    if (e < E) padded[e] = static_cast<int32_t>(before);
    carry += s_warp[kScanThreads / 32 - 1];
    __syncthreads();  // s_warp is rewritten by the next chunk
  }
  const bool any_bad = __syncthreads_or(bad) != 0;
  if (tid == 0) padded[E] = static_cast<int32_t>(carry);
  __syncthreads();
  if (any_bad) {
    for (int e = tid; e <= E; e += kScanThreads) padded[e] = -1;
  }
  if (tid == 0 && status != nullptr) *status = any_bad ? MXFP4_EOFFSETS : MXFP4_OK;
}



}  // namespace

cudaError_t launch_offsets(const int32_t* offsets, int32_t E, int64_t total_rows,
                           int32_t* scale_row_offsets, int32_t* status, cudaStream_t stream) {
  OffsetsParams q{};
  q.off = offsets;
  q.E = E;
  q.total_rows = total_rows;
  q.padded = scale_row_offsets;
  q.status = status;
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(q.dbg, kDbgOffsets, offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(q.dbg, kDbgPadded, scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(q.dbg, kDbgStatus, status, status ? 4 : 0);
#endif
  return launch_pdl(grouped_offsets_kernel, 1, kScanThreads, 0, stream, q);
}

cudaError_t launch_quantize(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes,
                            uint8_t* scales, bool f16, cudaStream_t stream) {
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
  p.n_units = static_cast<int32_t>(tiles * p.nKT);
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(p.dbg, kDbgX, x, ((M - 1) * ldx + K) * 2);
  debug_range(p.dbg, kDbgCodes, codes, M * (K / 2));
  debug_range(p.dbg, kDbgScales, scales, tiles * p.nKT * kChunkBytes);
#endif
  const bool v32 = vec32_ok(x, p.ldx_bytes);
  const auto kernel = f16 ? (v32 ? quantize_tiles_kernel<false, true, true>
                                 : quantize_tiles_kernel<false, false, true>)
                          : (v32 ? quantize_tiles_kernel<false, true>
                                 : quantize_tiles_kernel<false, false>);
  return launch_pdl(kernel, static_cast<unsigned>(p.n_units), kThreads, 0, stream, p);
}

cudaError_t launch_quantize_grouped(const void* x, int64_t total_rows, int64_t K,
                                    const int32_t* offsets, int32_t E, uint8_t* codes,
                                    uint8_t* scales, int32_t* scale_row_offsets,
                                    int32_t* status, int64_t bound_tiles, bool f16,
                                    cudaStream_t stream) {
  cudaError_t err = launch_offsets(offsets, E, total_rows, scale_row_offsets, status, stream);
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
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(p.dbg, kDbgX, x, total_rows * K * 2);
  debug_range(p.dbg, kDbgCodes, codes, total_rows * (K / 2));
  debug_range(p.dbg, kDbgScales, scales, bound_tiles * p.nKT * kChunkBytes);
  debug_range(p.dbg, kDbgOffsets, offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(p.dbg, kDbgPadded, scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4);
#endif
  const int64_t grid = bound_tiles * p.nKT;  // CTAs past the real padded total exit at once
  const bool v32 = vec32_ok(x, p.ldx_bytes);
  const auto kernel = f16 ? (v32 ? quantize_tiles_kernel<true, true, true>
                                 : quantize_tiles_kernel<true, false, true>)
                          : (v32 ? quantize_tiles_kernel<true, true>
                                 : quantize_tiles_kernel<true, false>);
  return launch_pdl(kernel, static_cast<unsigned>(grid), kThreads, 0, stream, p);
}

cudaError_t launch_quantize_grouped_gather(const void* x, int64_t num_src_rows, int64_t K,
                                           int64_t ldx, const int32_t* row_index,
                                           int64_t total_rows, const int32_t* offsets, int32_t E,
                                           uint8_t* codes, uint8_t* scales,
                                           int32_t* scale_row_offsets, int32_t* status,
                                           int64_t bound_tiles, bool f16, cudaStream_t stream) {
  cudaError_t err = launch_offsets(offsets, E, total_rows, scale_row_offsets, status, stream);
  if (err != cudaSuccess || E == 0 || bound_tiles == 0) return err;
  QuantizeParams p{};
  p.x = static_cast<const uint8_t*>(x);
  p.ldx_bytes = ldx * 2;
  p.M = total_rows;
  p.code_ld = K / 2;
  p.codes = codes;
  p.scales = scales;
  p.sK = static_cast<int32_t>(K / kBlock);
  p.nKT = (p.sK + kTileBlocks - 1) / kTileBlocks;
  p.offsets = offsets;
  p.padded = scale_row_offsets;
  p.E = E;
  p.row_index = row_index;
  p.num_src_rows = num_src_rows;
  p.status = status;
  p.n_mtiles = static_cast<int32_t>(bound_tiles);
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(p.dbg, kDbgX, x, ((num_src_rows - 1) * ldx + K) * 2);
  debug_range(p.dbg, kDbgCodes, codes, total_rows * (K / 2));
  debug_range(p.dbg, kDbgScales, scales, bound_tiles * p.nKT * kChunkBytes);
  debug_range(p.dbg, kDbgOffsets, offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(p.dbg, kDbgPadded, scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(p.dbg, kDbgRowIndex, row_index, total_rows * 4);
  debug_range(p.dbg, kDbgStatus, status, status ? 4 : 0);
#endif
  const int64_t grid = bound_tiles * ((p.nKT + kGatherChunkTiles - 1) / kGatherChunkTiles);
  const bool v32 = vec32_ok(x, p.ldx_bytes);
  const auto kernel = f16 ? (v32 ? quantize_gather_kernel<true, true>
                                 : quantize_gather_kernel<false, true>)
                          : (v32 ? quantize_gather_kernel<true, false>
                                 : quantize_gather_kernel<false, false>);
  return launch_pdl(kernel, static_cast<unsigned>(grid), kGatherThreads, 0, stream, p);
}

#ifdef MXFP4_DEBUG_BOUNDS
unsigned int debug_violations_quantize() {
  unsigned int v = 0, zero = 0;
  cudaMemcpyFromSymbol(&v, g_debug_violations, sizeof v);
  cudaMemcpyToSymbol(g_debug_violations, &zero, sizeof zero);
  return v;
}
#endif

}  // namespace mxfp4
