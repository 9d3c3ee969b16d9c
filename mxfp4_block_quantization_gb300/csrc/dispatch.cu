// dispatch.cu — the MoE dispatch fused into the grouped quantize, for
// sm_103a: the scatter (token -> rows, quantize_scatter_kernel, one warp per
// token row, read and quantized once), the gather through the same kernel
// (invert_bucket_kernel inverts the row -> token map first), the NVFP4
// experts quant as a scatter (nvfp4_scatter_kernel: codes and scales per
// route, each expert with its own global scale), and the staged forms, where
// the scale bytes are stored to a workspace (MXFP4: once per token; NVFP4:
// per route, by padded row) and tile_scales_kernel writes the 128x4-tiled
// scales in whole chunks.
//
// Method: vLLM PR #43557 page ("Fix the E8M0 scale computation in the MXFP4
// MoE CUTLASS kernel"), "Implementation breakdown" items 1 and 3 (the experts
// quant of the routed activations); the per-element and per-block steps are
// those of quantize.cu and nvfp4.cu (shared through mxfp4_device.cuh and
// nvfp4_device.cuh).
#include <cstdint>

#include <cuda_runtime.h>

#include "mxfp4_device.cuh"
#include "mxfp4_internal.h"
#include "nvfp4_device.cuh"
#include "../../include/mxfp4.h"

namespace mxfp4 {
namespace {

constexpr int kThreads = 256;  // scatter CTAs: 8 warps

// Buffer slots of the kernels' DebugRanges (bounds build).
enum : int {
  kDbgX = 0, kDbgCodes, kDbgScales, kDbgOffsets, kDbgPadded, kDbgRowIndex, kDbgStatus,
  kDbgWork  // the workspace: maps and staged scale words
};

constexpr int kInvertThreads = 256;
constexpr int kSmemSegs = 2048;  // up to this many segments are searched in shared memory

// Row -> padded row for the per-row map kernels.  With E <= cap the
// offsets and padded starts are copied to shared memory once per CTA (every
// thread of the block must call the constructor: it has a barrier) and each
// row's segment is a binary search there; otherwise find_segment on global
// memory.
struct SegmentSearch {
  int32_t* s_off;
  int32_t* s_pad;
  const int32_t* off;
  const int32_t* pad;
  int E;
  int total;
  bool smem;
  // s_off and s_pad hold cap + 1 entries each
  __device__ SegmentSearch(int32_t* so, int32_t* sp, const int32_t* o, const int32_t* pd, int e,
                           int tot, int cap = kSmemSegs)
      : s_off(so), s_pad(sp), off(o), pad(pd), E(e), total(tot), smem(e <= cap) {
    if (smem)
      for (int i = threadIdx.x; i <= E; i += blockDim.x) {
        s_off[i] = __ldg(off + i);
        s_pad[i] = __ldg(pad + i);
      }
    __syncthreads();
  }
  __device__ int rows_of(int e) const {  // n_e
    return smem ? s_off[e + 1] - s_off[e] : __ldg(off + e + 1) - __ldg(off + e);
  }
  __device__ int padded_start(int e) const { return smem ? s_pad[e] : __ldg(pad + e); }
  __device__ int padded_row(int v) const {  // v in [0, total)
    if (!smem) {
      const int e = find_segment(off, E, v, total);
      return __ldg(pad + e) + (v - __ldg(off + e));
    }
    int lo = 0, hi = E - 1;  // the largest e with o[e] <= v: its segment is not empty
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_off[mid] <= v) lo = mid; else hi = mid - 1;
    }
    return s_pad[lo] + (v - s_off[lo]);
  }
};

// Fused dispatch scatter: route j of token t lands on row dest_rows[t][j] of
// the expert-sorted batch.  Each warp owns one token: lanes 0..top_k-1
// resolve the token's routes once, then the warp streams the token row in
// passes of 512 elements (lane = 16 elements, 32 bytes), kScatterBatch
// passes' loads in flight at a time, quantizes each pass once and stores its
// codes to every destination as one contiguous 256-byte run per route (two
// full lines): each destination row's codes leave the SM as one stream and
// DRAM traffic is the algorithmic one.  The 4-byte scale word of each of the
// pass's four k-tiles (lanes 0, 8, 16, 24) goes either
//   direct: into the tiled layout of every route, under an L2 evict-last
//     policy (a 16-byte group of the tiled layout holds the words of four rows
//     32 apart, written by different warps at different times); the first E
//     CTAs zero the segments' pad rows; or
//   staged (kStaged): once per token into a workspace, from which
//     tile_scales_kernel writes the tiled scales in whole 512-byte chunks
//     (7.3 M scattered 4-byte stores on the MoE batch avoided).
// The gather through the scatter path uses the same kernel in bucket mode:
// warp t takes the rows invert_bucket_kernel put in token t's bucket, and
// spare warps walk the overflow list.
constexpr int kScatterWarps = kThreads / 32;  // tokens per CTA
constexpr int kScatterBatch = 4;              // passes with loads in flight together
constexpr int kScatterPass = 32 * kElems;     // elements per warp pass (4 k-tiles)

struct ScatterParams {
  const uint8_t* __restrict__ x;          // BF16 token rows
  int64_t ldx_bytes;                      // token row stride in bytes
  int64_t num_tokens;
  const int32_t* __restrict__ dest_rows;  // token-major: [num_tokens, top_k] row of every route,
                                          //   -1 = none; bucket mode: [num_tokens, kBucket]
  const int32_t* __restrict__ count;      // NULL: token-major; else bucket mode: warp t < T
                                          //   takes rows dest_rows[t*kBucket ..] of count[t]
  const int32_t* __restrict__ ovf_n;      //   (at most kBucket), warps past T walk the
  const int32_t* __restrict__ ovf_row;    //   overflow list: ovf_row[j] of token ovf_tok[j],
  const int32_t* __restrict__ ovf_tok;    //   j < *ovf_n, n_ovf_warps warps in all
  int32_t n_ovf_warps;
  int32_t top_k;
  int32_t E;
  int64_t total_rows;                     // rows of the expert-sorted batch
  int64_t code_ld;                        // K/2
  uint8_t* __restrict__ codes;
  uint8_t* __restrict__ scales;
  const int32_t* __restrict__ offsets;    // [E+1] row offsets of the segments
  const int32_t* __restrict__ padded;     // [E+1] padded row starts
  int32_t* status;                        // may be NULL
  uint32_t* __restrict__ stage;           // kStaged: [num_tokens, stage_ld(nKT)] scale words
                                          //   of every token, tiled by tile_scales_kernel
  int32_t pad_ctas;                       // leading CTAs that zero pad scale rows (E or 0)
  int32_t sK;
  int32_t nKT;
  int32_t map_ctas;                       // kStaged, token-major: the next CTAs write tok1,
  int32_t* __restrict__ tok1;             //   the token + 1 of every padded row (-1: pad row)
  int64_t code_rows;                      // codes are written for rows < code_rows only (the
                                          //   rows past it hold a borrowed workspace)
#ifdef MXFP4_DEBUG_BOUNDS
  DebugRanges dbg;                        // slots as in QuantizeParams (kDbgRowIndex: dest_rows)
#endif
};

// Row stride, in 4-byte words, of the staged per-token scale words: nKT
// rounded up to 16 bytes so that the tile kernel reads them as uint4.
__host__ __device__ __forceinline__ int64_t stage_ld(int nKT) { return (nKT + 3) & ~3; }

// Byte offset of the scale word (4 scale columns of one k-tile) of padded row
// `prow` in k-tile 0; k-tile kt adds kt * 512.
__device__ __forceinline__ int64_t scale_word_base(int prow, int nKT) {
  return static_cast<int64_t>(prow >> 7) * nKT * kChunkBytes + (prow & 31) * 16 +
         ((prow & 127) >> 5) * 4;
}

// One warp: token row t, quantized once, to the nr (<= 32) rows dsts[0..nr).
template <bool kVec32, bool kF16, bool kStaged>
__device__ __forceinline__ void scatter_token(const ScatterParams& p, int64_t t,
                                              const int32_t* dsts, int nr, int warp, int lane,
                                              int64_t (*s_code)[MXFP4_SCATTER_MAX_TOP_K],
                                              int64_t (*s_scale)[MXFP4_SCATTER_MAX_TOP_K]) {
  // routes, one per lane
  int64_t co = -1, so = -1;
  bool bad = false;
  if (lane < nr) {
    const int32_t* dp = dsts + lane;
    const int32_t v = MXFP4_IN_BOUNDS(p, kDbgRowIndex, dp, 4) ? __ldg(dp) : -1;
    if (v >= 0 && v < p.total_rows) {
      co = v < p.code_rows ? static_cast<int64_t>(v) * p.code_ld : -1;
      if constexpr (!kStaged) {
        const int e = find_segment(p.offsets, p.E, v, static_cast<int>(p.total_rows));
        so = scale_word_base(__ldg(p.padded + e) + (v - __ldg(p.offsets + e)), p.nKT);
      }
    } else {
      bad = v != -1;
    }
  }
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && p.status != nullptr &&
      MXFP4_IN_BOUNDS(p, kDbgStatus, p.status, 4))
    atomicExch(p.status, MXFP4_EINDEX);
  s_code[warp][lane] = co;
  // staged: no per-route scale words; slot 0 holds the token's stage row instead
  s_scale[warp][lane] = kStaged ? reinterpret_cast<int64_t>(p.stage + t * stage_ld(p.nKT)) : so;
  __syncwarp();

  const uint8_t* xrow = p.x + t * p.ldx_bytes + lane * (kElems * 2);
  const int n_pass = (p.sK + 15) / 16;  // 16 blocks per pass
  const uint64_t keep = l2_evict_last_policy();
  for (int p0 = 0; p0 < n_pass; p0 += kScatterBatch) {
    uint4 v[kScatterBatch][2];
#pragma unroll
    for (int b = 0; b < kScatterBatch; ++b) {
      v[b][0] = v[b][1] = make_uint4(0u, 0u, 0u, 0u);
      const int pass = p0 + b;
      const uint8_t* xp = xrow + static_cast<int64_t>(pass) * (kScatterPass * 2);
      if (pass < n_pass && pass * 16 + (lane >> 1) < p.sK &&
          MXFP4_IN_BOUNDS(p, kDbgX, xp, 32))
        load32<kVec32>(xp, v[b]);
    }
    uint2 code[kScatterBatch];
    uint32_t word[kScatterBatch];
#pragma unroll
    for (int b = 0; b < kScatterBatch; ++b) {
      const uint32_t s = lane_block_scale<kF16>(v[b]);
      code[b] = lane_codes<kF16>(v[b], s);
      // scale word of k-tile (p0+b)*4 + lane/8: the s of lanes +0, +2, +4, +6
      word[b] = s | (__shfl_down_sync(0xFFFFFFFFu, s, 2) << 8) |
                (__shfl_down_sync(0xFFFFFFFFu, s, 4) << 16) |
                (__shfl_down_sync(0xFFFFFFFFu, s, 6) << 24);
    }
    const int64_t cofs = static_cast<int64_t>(p0) * (kScatterPass / 2) + lane * (kElems / 2);
    const int kt0 = p0 * 4 + (lane >> 3);
    if (kStaged && (lane & 7) == 0) {
      // the token's words once (every warp of a token stores the same values)
      uint32_t* const srow = reinterpret_cast<uint32_t*>(s_scale[warp][0]);
#pragma unroll
      for (int b = 0; b < kScatterBatch; ++b) {
        const int kt = kt0 + 4 * b;
        uint32_t* const sp = srow + kt;
        if (kt < p.nKT && MXFP4_IN_BOUNDS(p, kDbgWork, sp, 4)) st_keep_u32(sp, word[b], keep);
      }
    }
    for (int j = 0; j < nr; ++j) {
      const int64_t c = s_code[warp][j];
      const int64_t w = s_scale[warp][j];
#pragma unroll
      for (int b = 0; b < kScatterBatch; ++b) {
        const int pass = p0 + b;
        uint8_t* const cp = p.codes + c + cofs + b * (kScatterPass / 2);
        if (c >= 0 && pass * 16 + (lane >> 1) < p.sK && MXFP4_IN_BOUNDS(p, kDbgCodes, cp, 8))
          st_stream_v2(cp, code[b]);
        if constexpr (!kStaged) {
          const int kt = kt0 + 4 * b;
          uint8_t* const wp = p.scales + w + static_cast<int64_t>(kt) * kChunkBytes;
          if (w >= 0 && (lane & 7) == 0 && kt < p.nKT && MXFP4_IN_BOUNDS(p, kDbgScales, wp, 4))
            st_keep_u32(wp, word[b], keep);
        }
      }
    }
  }
  __syncwarp();  // s_code / s_scale are rewritten by the warp's next token
}

// Map CTA m of the staged token-major scatter: the token + 1 (or the padded
// row + 1) of every padded row a route lands on, and -1 for the pad rows of
// every segment (rows no route targets keep the 0 of the memset).  The tile
// kernel reads the map after this launch has completed.  The offsets and
// padded starts (up to kMapSegs + 1 each) reuse the warps' route arrays.
constexpr int kMapSegs = 511;
static_assert((kMapSegs + 1) * 4 == kScatterWarps * MXFP4_SCATTER_MAX_TOP_K * 8,
              "one segment array fills one route array");
// kPadOnly: write the pad rows only (the NVFP4 scatter's token warps write
// their own routes' entries, each pointing at the row of staged scale bytes
// the route reads).
template <bool kPadOnly = false, typename P>
__device__ __forceinline__ void scatter_route_map(const P& p, int m, int32_t* s_off,
                                                  int32_t* s_pad) {
  const SegmentSearch seg(s_off, s_pad, p.offsets, p.padded, p.E,
                          static_cast<int>(p.total_rows), kMapSegs);
  const int64_t gid = static_cast<int64_t>(m) * kThreads + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(p.map_ctas) * kThreads;
  // the pad rows: item k is pad slot k % 128 of segment k / 128, so that
  // consecutive threads store consecutive rows of one segment
  for (int64_t k = gid; k < static_cast<int64_t>(p.E) * kTileRows; k += stride) {
    const int e = static_cast<int>(k / kTileRows);
    const int i = static_cast<int>(k % kTileRows);
    const int n = seg.rows_of(e);
    const int npad = (n + kTileRows - 1) / kTileRows * kTileRows - n;
    if (i >= npad) continue;
    int32_t* const tp = p.tok1 + seg.padded_start(e) + n + i;
    if (MXFP4_IN_BOUNDS(p, kDbgWork, tp, 4)) *tp = -1;
  }
  if constexpr (kPadOnly) return;
  const int64_t n_routes = p.num_tokens * p.top_k;
  for (int64_t i = gid; i < n_routes; i += stride) {
    const int32_t* dp = p.dest_rows + i;
    const int32_t v = MXFP4_IN_BOUNDS(p, kDbgRowIndex, dp, 4) ? __ldg(dp) : -1;
    if (v < 0 || v >= p.total_rows) continue;  // the token warps report bad entries
    const int prow = seg.padded_row(v);
    int32_t* const tp = p.tok1 + prow;
    if (MXFP4_IN_BOUNDS(p, kDbgWork, tp, 4)) *tp = static_cast<int32_t>(i / p.top_k) + 1;
  }
}

// Overflow entry j (bucket mode): its token and row; false past the list.
__device__ __forceinline__ bool overflow_entry(const ScatterParams& p, int64_t j, int64_t& t,
                                               const int32_t*& dsts) {
  if (!MXFP4_IN_BOUNDS(p, kDbgWork, p.ovf_n, 4)) return false;
  const int64_t n = __ldg(p.ovf_n);
  if (j >= n || j >= p.total_rows || !MXFP4_IN_BOUNDS(p, kDbgWork, p.ovf_tok + j, 4))
    return false;
  t = __ldg(p.ovf_tok + j);
  dsts = p.ovf_row + j;
  return true;
}

template <bool kVec32, bool kF16, bool kStaged>
__global__ void __launch_bounds__(kThreads, kStaged ? 5 : 0) quantize_scatter_kernel(const ScatterParams p) {
  __shared__ int64_t s_code[kScatterWarps][MXFP4_SCATTER_MAX_TOP_K];   // d * K/2, or -1
  __shared__ int64_t s_scale[kScatterWarps][MXFP4_SCATTER_MAX_TOP_K];  // word base, or -1
  __shared__ int64_t s_next[kScatterWarps];  // overflow warps: their current entry

  pdl_wait();
  pdl_release();

  if (!MXFP4_IN_BOUNDS(p, kDbgPadded, p.padded, (p.E + 1) * 4) ||
      !MXFP4_IN_BOUNDS(p, kDbgOffsets, p.offsets, (p.E + 1) * 4))
    return;
  const int total_padded = __ldg(p.padded + p.E);
  if (total_padded < 0) return;  // rejected offsets

  if (static_cast<int>(blockIdx.x) < p.pad_ctas) {
    // pad rows [n, ceil128(n)) of expert e: zero scale words, row-fastest
    const int e = blockIdx.x;
    const int n = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
    const int npad = ((n + kTileRows - 1) / kTileRows) * kTileRows - n;
    const int P0 = __ldg(p.padded + e) + n;
    const uint64_t keep = l2_evict_last_policy();
    for (int i = threadIdx.x; i < npad * p.nKT; i += kThreads) {
      const int kt = i / npad;
      uint8_t* wp = p.scales + scale_word_base(P0 + (i - kt * npad), p.nKT) + kt * kChunkBytes;
      if (MXFP4_IN_BOUNDS(p, kDbgScales, wp, 4)) st_keep_u32(wp, 0u, keep);
    }
    return;
  }

  if constexpr (kStaged) {
    const int m = static_cast<int>(blockIdx.x) - p.pad_ctas;
    if (m < p.map_ctas) {  // uniform over the block
      scatter_route_map(p, m, reinterpret_cast<int32_t*>(&s_code[0][0]),
                        reinterpret_cast<int32_t*>(&s_scale[0][0]));
      return;
    }
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int lead = p.pad_ctas + (kStaged ? p.map_ctas : 0);  // CTAs before the token warps
  const int64_t w_id = static_cast<int64_t>(blockIdx.x - lead) * kScatterWarps + warp;
  // whole warps return below; there is no block-wide barrier after this point
  int64_t t;
  const int32_t* dsts;
  int nr;
  if (p.count == nullptr) {  // token-major: warp = token, top_k routes
    if (w_id >= p.num_tokens) return;
    t = w_id;
    dsts = p.dest_rows + w_id * p.top_k;
    nr = p.top_k;
  } else if (w_id < p.num_tokens) {  // bucket mode: the token's first kBucket rows
    if (!MXFP4_IN_BOUNDS(p, kDbgWork, p.count + w_id, 4)) return;
    const int c = __ldg(p.count + w_id);
    if (c <= 0) return;
    t = w_id;
    dsts = p.dest_rows + w_id * MXFP4_SCATTER_MAX_TOP_K;
    nr = c < MXFP4_SCATTER_MAX_TOP_K ? c : MXFP4_SCATTER_MAX_TOP_K;
  } else {  // bucket mode: the overflow list, one row per entry, warp-strided
    const int64_t j = w_id - p.num_tokens;
    if (!overflow_entry(p, j, t, dsts)) return;
    s_next[warp] = j;
    nr = 1;
  }
  for (;;) {
    scatter_token<kVec32, kF16, kStaged>(p, t, dsts, nr, warp, lane, s_code, s_scale);
    // only overflow warps go on; their cursor is kept in shared memory so that
    // nothing stays live across the body above
    if (p.count == nullptr ||
        static_cast<int64_t>(blockIdx.x - p.pad_ctas - (kStaged ? p.map_ctas : 0)) *
                    kScatterWarps + warp < p.num_tokens)
      return;
    const int64_t j = s_next[warp] + p.n_ovf_warps;
    if (!overflow_entry(p, j, t, dsts)) return;
    __syncwarp();
    s_next[warp] = j;
  }
}

// The gather without a caller workspace borrows the last rows of its own
// codes output as the workspace: the kernels above leave those rows' codes
// unwritten (code_rows), and gather_row_codes_kernel writes them last, once
// the workspace is no longer read.  clear_words_kernel zeroes the workspace's
// counters only for valid offsets, so that rejected offsets still leave the
// outputs untouched.
__global__ void __launch_bounds__(kThreads) clear_words_kernel(const int32_t* padded, int32_t E,
                                                              uint4* words, int64_t n16) {
  pdl_wait();
  pdl_release();
  if (__ldg(padded + E) < 0) return;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n16;
       i += static_cast<int64_t>(gridDim.x) * kThreads)
    words[i] = make_uint4(0u, 0u, 0u, 0u);
}

struct RowCodesParams {
  const uint8_t* __restrict__ x;          // 16-bit source rows
  int64_t ldx_bytes;
  int64_t num_src_rows;
  const int32_t* __restrict__ row_index;  // [R] source row of every row
  int64_t r0;                             // rows [r0, R) get their codes here
  int64_t total_rows;                     // R
  uint8_t* __restrict__ codes;
  int64_t code_ld;
  const int32_t* __restrict__ padded;
  int32_t E;
  int32_t sK;
#ifdef MXFP4_DEBUG_BOUNDS
  DebugRanges dbg;  // kDbgX, kDbgCodes, kDbgPadded, kDbgRowIndex
#endif
};

// Rows r in [r0, R) get the codes of source row row_index[r] (zero codes for
// an index out of range).  One warp per row and group of kRowGroup passes of
// 512 elements: the group's loads are issued first, so that a batch of a few
// thousand rows still keeps enough loads in flight.
constexpr int kRowGroup = 4;

template <bool kVec32, bool kF16>
__global__ void __launch_bounds__(kThreads) gather_row_codes_kernel(const RowCodesParams p) {
  pdl_wait();
  pdl_release();
  if (!MXFP4_IN_BOUNDS(p, kDbgPadded, p.padded + p.E, 4) || __ldg(p.padded + p.E) < 0) return;
  const int lane = threadIdx.x & 31;
  const int n_pass = (p.sK + 15) / 16;
  const int n_grp = (n_pass + kRowGroup - 1) / kRowGroup;
  const int64_t w = static_cast<int64_t>(blockIdx.x) * kScatterWarps + (threadIdx.x >> 5);
  const int64_t r = p.r0 + w / n_grp;
  if (r >= p.total_rows) return;  // whole warp
  const int pass0 = static_cast<int>(w % n_grp) * kRowGroup;
  const int32_t* ip = p.row_index + r;
  const int32_t t = MXFP4_IN_BOUNDS(p, kDbgRowIndex, ip, 4) ? __ldg(ip) : -1;
  const bool valid = t >= 0 && t < p.num_src_rows;
  const uint8_t* xrow = p.x + (valid ? t : 0) * p.ldx_bytes + lane * (kElems * 2);
  uint8_t* crow = p.codes + r * p.code_ld + lane * (kElems / 2);
  uint4 v[kRowGroup][2];
#pragma unroll
  for (int i = 0; i < kRowGroup; ++i) {
    const int pass = pass0 + i;
    v[i][0] = make_uint4(0u, 0u, 0u, 0u);
    v[i][1] = make_uint4(0u, 0u, 0u, 0u);
    const uint8_t* xp = xrow + static_cast<int64_t>(pass) * (kScatterPass * 2);
    if (valid && pass * 16 + (lane >> 1) < p.sK && MXFP4_IN_BOUNDS(p, kDbgX, xp, 32))
      load32<kVec32>(xp, v[i]);
  }
#pragma unroll
  for (int i = 0; i < kRowGroup; ++i) {
    const int pass = pass0 + i;
    const uint32_t sc = lane_block_scale<kF16>(v[i]);  // all lanes: the pair shares a shuffle
    const uint2 code = lane_codes<kF16>(v[i], sc);
    uint8_t* const cp = crow + static_cast<int64_t>(pass) * (kScatterPass / 2);
    if (pass * 16 + (lane >> 1) < p.sK && MXFP4_IN_BOUNDS(p, kDbgCodes, cp, 8))
      st_stream_v2(cp, code);
  }
}

// NVFP4 experts quant with the MoE dispatch as a scatter: route j of token t
// lands on row dest_rows[t][j] of the expert-sorted batch, whose segment e
// has global scale g[e].  One warp per token: the row is read once, in passes
// of 512 elements (lane = one 16-element block), and each block's max and
// q = vecMax / 6 are taken once; then, per route, the block's E4M3 byte
// (g[e] * q), inverse scale and codes with that route's global scale (a
// token's codes differ per expert), or once for all routes when the token's
// experts share one global scale.  Codes leave as one 256-byte run per route
// and pass.  The scale bytes go either
//   direct: as the 4-byte word of each k-tile (4 lanes) into the tiled layout
//     of every route, under an L2 evict-last policy (14.7 M scattered words on
//     the MoE batch); the first E CTAs zero the segments' pad rows; or
//   staged (kStaged): as one 32-byte run per route and pass into the route's
//     padded row of a workspace, which tile_scales_kernel then writes to the
//     tiled layout whole.  Each token warp records, for each route, the
//     workspace row its bytes are in (+1): its own, or for a token whose
//     routes share one scale the first route's, the only row it stages.  The
//     first map_ctas CTAs mark the pad rows -1 beside the token warps.
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
  int32_t pad_ctas;                       // direct: E CTAs zero the pad rows
  int32_t map_ctas;                       // staged: CTAs writing tok1
  int32_t* __restrict__ tok1;             // staged: [padded rows] padded row + 1, -1 pad row
  uint8_t* __restrict__ stage;            // staged: [padded rows, 4 * stage_ld(nKT)] scale bytes
#ifdef MXFP4_DEBUG_BOUNDS
  DebugRanges dbg;                        // kDbg slots; kDbgWork: the workspace
  DebugRanges dbg_g;                      // slot 0: the global scales
#endif
};

#ifdef MXFP4_DEBUG_BOUNDS
#define MXFP4_IN_BOUNDS_G(params, ptr, bytes) \
  ::mxfp4::debug_in_bounds((params).dbg_g, 0, (ptr), (bytes))
#else
#define MXFP4_IN_BOUNDS_G(params, ptr, bytes) true
#endif

constexpr int kNvScBatch = 2;  // passes with loads in flight together (4 CTAs per SM)

// Byte offset of the scale word of padded row prow in k-tile 0 of the tiled
// layout (k-tile kt adds kt * 512) — or, staged, of its workspace row.
template <bool kStaged>
__device__ __forceinline__ int64_t nv_row_base(int prow, int nKT) {
  if constexpr (kStaged) return static_cast<int64_t>(prow) * stage_ld(nKT) * 4;
  return scale_word_base(prow, nKT);
}

__device__ __forceinline__ void st_keep_u8(void* p, uint32_t v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.u8 [%0], %1, %2;" ::"l"(p), "r"(v), "l"(policy)
               : "memory");
}

template <bool kVec32, bool kF16, bool kStaged>
__global__ void __launch_bounds__(kThreads, 4) nvfp4_scatter_kernel(const Nvfp4ScatterParams p) {
  __shared__ int64_t s_code[kScatterWarps][MXFP4_SCATTER_MAX_TOP_K];  // d * K/2, or -1
  __shared__ int64_t s_word[kScatterWarps][MXFP4_SCATTER_MAX_TOP_K];  // scale row base
  __shared__ float s_g[kScatterWarps][MXFP4_SCATTER_MAX_TOP_K];       // the route's scale

  pdl_wait();
  pdl_release();

  if (!MXFP4_IN_BOUNDS(p, kDbgPadded, p.padded, (p.E + 1) * 4) ||
      !MXFP4_IN_BOUNDS(p, kDbgOffsets, p.offsets, (p.E + 1) * 4))
    return;
  if (__ldg(p.padded + p.E) < 0) return;  // rejected offsets: nothing is written

  if (static_cast<int>(blockIdx.x) < p.pad_ctas) {
    // pad rows [n, ceil128(n)) of segment e: zero scale words, row-fastest
    const int e = blockIdx.x;
    const int n = __ldg(p.offsets + e + 1) - __ldg(p.offsets + e);
    const int npad = ((n + kTileRows - 1) / kTileRows) * kTileRows - n;
    const int P0 = __ldg(p.padded + e) + n;
    const uint64_t keep = l2_evict_last_policy();
    for (int i = threadIdx.x; i < npad * p.nKT; i += kThreads) {
      const int kt = i / npad;
      uint8_t* wp = p.scales + scale_word_base(P0 + (i - kt * npad), p.nKT) + kt * kChunkBytes;
      if (MXFP4_IN_BOUNDS(p, kDbgScales, wp, 4)) st_keep_u32(wp, 0u, keep);
    }
    return;
  }
  if constexpr (kStaged) {
    const int m = static_cast<int>(blockIdx.x) - p.pad_ctas;
    if (m < p.map_ctas) {  // uniform over the block
      scatter_route_map<true>(p, m, reinterpret_cast<int32_t*>(&s_code[0][0]),
                              reinterpret_cast<int32_t*>(&s_word[0][0]));
      return;
    }
  }

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int lead = p.pad_ctas + (kStaged ? p.map_ctas : 0);
  const int64_t t = static_cast<int64_t>(blockIdx.x - lead) * kScatterWarps + warp;
  if (t >= p.num_tokens) return;  // whole warp; no block-wide barrier below

  // routes, one per lane
  int64_t co = -1, wo = -1;
  int32_t prow = -1;
  float ge = 0.0f;
  bool bad = false;
  if (lane < p.top_k) {
    const int32_t* dp = p.dest_rows + t * p.top_k + lane;
    const int32_t v = MXFP4_IN_BOUNDS(p, kDbgRowIndex, dp, 4) ? __ldg(dp) : -1;
    if (v >= 0 && v < p.total_rows) {
      const int e = find_segment(p.offsets, p.E, v, static_cast<int>(p.total_rows));
      co = static_cast<int64_t>(v) * p.code_ld;
      prow = __ldg(p.padded + e) + (v - __ldg(p.offsets + e));
      wo = nv_row_base<kStaged>(prow, p.nKT);
      ge = MXFP4_IN_BOUNDS_G(p, p.g + e, 4) ? __ldg(p.g + e) : 0.0f;
    } else {
      bad = v != -1;
    }
  }
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0 && p.status != nullptr &&
      MXFP4_IN_BOUNDS(p, kDbgStatus, p.status, 4))
    atomicExch(p.status, MXFP4_EINDEX);
  s_code[warp][lane] = co;
  s_word[warp][lane] = wo;
  s_g[warp][lane] = ge;
  __syncwarp();

  // A token whose routes all land in experts of one global scale (the same
  // bits) has the same bytes and codes on every route: those are computed
  // once per pass and stored to each route.  Any other token takes the
  // per-route loop.  Decided once per token, outside the route loops.
  const unsigned routed = __ballot_sync(0xFFFFFFFFu, co >= 0);
  if (routed == 0u) return;  // whole warp: nothing to write
  const int first = __ffs(static_cast<int>(routed)) - 1;  // the first route
  const float g0 = __shfl_sync(0xFFFFFFFFu, ge, first);
  const bool one_scale =
      __all_sync(0xFFFFFFFFu, co < 0 || __float_as_uint(ge) == __float_as_uint(g0));
  if constexpr (kStaged) {
    // each route's map entry: the staged row its scale bytes are read from,
    // + 1; with one scale the token stages them once, in its first route's row
    const int32_t prow0 = __shfl_sync(0xFFFFFFFFu, prow, first);
    int32_t* const tp = p.tok1 + prow;
    if (co >= 0 && MXFP4_IN_BOUNDS(p, kDbgWork, tp, 4)) *tp = (one_scale ? prow0 : prow) + 1;
  }

  const uint8_t* xrow = p.x + t * p.ldx_bytes + lane * 32;
  const int n_pass = (p.sK + 31) / 32;  // 32 blocks per pass
  const uint64_t keep = l2_evict_last_policy();
  // the stores of pass p0 + b for the route with codes at c and scale row w
  auto put = [&](int64_t c, int64_t w, int p0, int b, uint32_t byte, uint2 code, bool stage) {
    const int pass = p0 + b;
    const int blk = pass * 32 + lane;
    uint8_t* const cp = p.codes + c + static_cast<int64_t>(blk) * 8;
    if (pass < n_pass && blk < p.sK && MXFP4_IN_BOUNDS(p, kDbgCodes, cp, 8))
      st_stream_v2(cp, code);
    if constexpr (kStaged) {
      // the route's scale bytes, 32 per pass, into its workspace row (zero
      // for the pad columns past sK)
      uint8_t* const bp = p.stage + w + blk;
      if (stage && pass < n_pass && blk < 4 * p.nKT && MXFP4_IN_BOUNDS(p, kDbgWork, bp, 1))
        st_keep_u8(bp, byte, keep);
    } else {
      // scale word of k-tile pass*8 + lane/4: the bytes of lanes +0..+3
      const uint32_t word = byte | (__shfl_down_sync(0xFFFFFFFFu, byte, 1) << 8) |
                            (__shfl_down_sync(0xFFFFFFFFu, byte, 2) << 16) |
                            (__shfl_down_sync(0xFFFFFFFFu, byte, 3) << 24);
      const int kt = pass * 8 + (lane >> 2);
      uint8_t* const wp = p.scales + w + static_cast<int64_t>(kt) * kChunkBytes;
      if (pass < n_pass && (lane & 3) == 0 && kt < p.nKT && MXFP4_IN_BOUNDS(p, kDbgScales, wp, 4))
        st_keep_u32(wp, word, keep);
    }
  };
  for (int p0 = 0; p0 < n_pass; p0 += kNvScBatch) {
    uint4 v[kNvScBatch][2];
    float q[kNvScBatch];
#pragma unroll
    for (int b = 0; b < kNvScBatch; ++b) {
      v[b][0] = v[b][1] = make_uint4(0u, 0u, 0u, 0u);
      const int blk = (p0 + b) * 32 + lane;
      const uint8_t* xp = xrow + static_cast<int64_t>(p0 + b) * 1024;
      if (p0 + b < n_pass && blk < p.sK && MXFP4_IN_BOUNDS(p, kDbgX, xp, 32))
        load32<kVec32>(xp, v[b]);
    }
#pragma unroll
    for (int b = 0; b < kNvScBatch; ++b) q[b] = nv_block_q<kF16>(v[b]);
    if (one_scale) {  // uniform over the warp
      uint32_t bytes[kNvScBatch];
      uint2 codes[kNvScBatch];
#pragma unroll
      for (int b = 0; b < kNvScBatch; ++b) {
        bytes[b] = cvt_e4m3_satfinite(g0 * q[b]);
        codes[b] = nv_codes<kF16>(v[b], bytes[b],
                                  bytes[b] != 0u ? g0 / e4m3_to_f32(bytes[b]) : 0.0f);
      }
      for (int j = 0; j < p.top_k; ++j) {
        const int64_t c = s_code[warp][j];
        if (c < 0) continue;  // the same for every lane of the warp
        const int64_t w = s_word[warp][j];
#pragma unroll
        for (int b = 0; b < kNvScBatch; ++b) put(c, w, p0, b, bytes[b], codes[b], j == first);
      }
    } else {
      for (int j = 0; j < p.top_k; ++j) {
        const int64_t c = s_code[warp][j];
        if (c < 0) continue;
        const int64_t w = s_word[warp][j];
        const float g = s_g[warp][j];
#pragma unroll
        for (int b = 0; b < kNvScBatch; ++b) {
          const uint32_t byte = cvt_e4m3_satfinite(g * q[b]);
          put(c, w, p0, b, byte,
              nv_codes<kF16>(v[b], byte, byte != 0u ? g / e4m3_to_f32(byte) : 0.0f), true);
        }
      }
    }
  }
}

// Tiled scales of the gathered or scattered batch from the staged per-token
// words: one CTA per padded 128-row tile.  Padded row pr takes the words of
// token tok1[pr] - 1 (for the gather written by invert_bucket_kernel for row
// o[e] + pr - P[e] of segment e, for the scatter by the map CTAs of the
// scatter launch; in the NVFP4 scatter the staged rows are rows of scale
// bytes, one per route or one per token, written by the token warps).  In
// the gather, pad rows and rows whose index is out of
// range keep tok1 = 0 and get zero words; in the scatter, pad rows are marked
// -1 and get zero words, and rows that no route targets (0) keep the words
// they held.  The words pass through shared memory so that every 512-byte
// chunk is written whole, 16 bytes per thread, instead of 4-byte words
// scattered over the chunks.  One CTA covers one tile and kTileCols of its
// k-tiles (one load phase, one barrier, one store phase): the several CTAs of
// a tile and their neighbours on an SM are in different phases at any time,
// so the loads of some overlap the stores of others.
struct TileScalesParams {
  const int32_t* __restrict__ tok1;       // [grid * 128] token + 1 of every padded row, 0: none,
                                          //   -1: pad row (kKeep only)
  const uint32_t* __restrict__ stage;     // [T, stage_ld(nKT)], 16-byte aligned
  uint8_t* __restrict__ scales;
  const int32_t* __restrict__ padded;
  int32_t E;
  int32_t nKT;
  int32_t n_kc;                           // CTAs per tile: ceil(nKT / kTileCols)
#ifdef MXFP4_DEBUG_BOUNDS
  DebugRanges dbg;  // kDbgScales, kDbgPadded, kDbgRowIndex (tok1), kDbgWork (stage)
#endif
};

// 128 threads and 16 k-tiles (9 KB of shared memory) per CTA, up to twelve
// CTAs per SM.
constexpr int kTileThreads = 128;
constexpr int kTileCols = 16;                                  // k-tiles per CTA
constexpr int kTileQuadsPerRow = kTileCols / 4;                // 16-byte quads of a row
constexpr int kTileRowStep = kTileThreads / kTileQuadsPerRow;  // rows per load step
constexpr int kTileQuads = kTileRows / kTileRowStep;           // uint4 loads per thread
static_assert(kTileRows % kTileRowStep == 0 && kTileRows <= kTileThreads,
              "tile_scales_kernel: whole load steps, one token per thread");

// kKeep: rows with tok1 == 0 keep their words (the scatter); otherwise they
// get zero words like pad rows (the gather).
template <bool kKeep>
__global__ void __launch_bounds__(kTileThreads, 12) tile_scales_kernel(const TileScalesParams p) {
  __shared__ uint32_t s_w[kTileRows][kTileCols + 1];  // odd stride: conflict-free columns
  __shared__ int32_t s_tok[kTileRows];
  __shared__ const uint32_t* s_row[kTileRows];        // the row's staged words, or NULL

  pdl_wait();
  pdl_release();

  if (!MXFP4_IN_BOUNDS(p, kDbgPadded, p.padded + p.E, 4)) return;
  const int tile_id = static_cast<int>(blockIdx.x) / p.n_kc;
  const int c0 = (static_cast<int>(blockIdx.x) - tile_id * p.n_kc) * kTileCols;
  const int pr0 = tile_id * kTileRows;
  // both loads in flight together: the tile's tokens and the padded total
  int32_t t1 = 0;
  if (threadIdx.x < kTileRows) {
    const int32_t* tp = p.tok1 + pr0 + threadIdx.x;
    if (MXFP4_IN_BOUNDS(p, kDbgRowIndex, tp, 4)) t1 = __ldg(tp);
  }
  const int total_padded = __ldg(p.padded + p.E);
  if (total_padded < 0 || pr0 >= total_padded) return;  // whole CTA: nothing past P[E]
  if (threadIdx.x < kTileRows) {
    s_tok[threadIdx.x] = t1 - 1;
    s_row[threadIdx.x] =
        t1 > 0 ? p.stage + static_cast<int64_t>(t1 - 1) * stage_ld(p.nKT) : nullptr;
  }
  __syncthreads();

  uint8_t* const tile = p.scales + static_cast<int64_t>(tile_id) * p.nKT * kChunkBytes;
  const int qd = threadIdx.x % kTileQuadsPerRow;  // this thread's quad: words 4qd .. 4qd+3
  const int rb = threadIdx.x / kTileQuadsPerRow;  // and its rows rb, rb + kTileRowStep, ...
  {
    const int cw = p.nKT - c0 < kTileCols ? p.nKT - c0 : kTileCols;
    const bool in_row = 4 * qd < cw;
    // every load of the pass in flight before the first shared-memory store
    uint4 v[kTileQuads];
#pragma unroll
    for (int j = 0; j < kTileQuads; ++j) {
      const int r = rb + kTileRowStep * j;
      const uint32_t* const rp = s_row[r];
      v[j] = make_uint4(0u, 0u, 0u, 0u);
      if (rp != nullptr && in_row) {
        const uint32_t* sp = rp + c0 + 4 * qd;
        if (MXFP4_IN_BOUNDS(p, kDbgWork, sp, 16)) v[j] = __ldg(reinterpret_cast<const uint4*>(sp));
      } else if (kKeep && in_row && s_tok[r] == -1) {
        // an untargeted row keeps its words: read them back (this pass's
        // chunks are written only after the barrier below)
        const uint8_t* op = tile + static_cast<int64_t>(c0 + 4 * qd) * kChunkBytes +
                            (r & 31) * 16 + (r >> 5) * 4;
        uint32_t w4[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (c0 + 4 * qd + i < p.nKT && MXFP4_IN_BOUNDS(p, kDbgScales, op + i * kChunkBytes, 4))
            w4[i] = *reinterpret_cast<const uint32_t*>(op + i * kChunkBytes);
        v[j] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
    }
    if (in_row) {
#pragma unroll
      for (int j = 0; j < kTileQuads; ++j) {
        uint32_t* const w = &s_w[rb + kTileRowStep * j][4 * qd];  // words past cw: never read
        w[0] = v[j].x;
        w[1] = v[j].y;
        w[2] = v[j].z;
        w[3] = v[j].w;
      }
    }
    __syncthreads();
    // piece (c, o): rows o, o+32, o+64, o+96 of k-tile c0 + c, bytes o*16 of its chunk
    for (int i = threadIdx.x; i < cw * 32; i += kTileThreads) {
      const int c = i >> 5;
      const int o = i & 31;
      uint8_t* const dp = tile + static_cast<int64_t>(c0 + c) * kChunkBytes + o * 16;
      if (MXFP4_IN_BOUNDS(p, kDbgScales, dp, 16))
        st_stream_v4(dp, make_uint4(s_w[o][c], s_w[o + 32][c], s_w[o + 64][c], s_w[o + 96][c]));
    }
  }
}

// The tile kernel's launch over `tiles` padded tiles.
cudaError_t launch_tile_scales(bool keep, TileScalesParams ts, int64_t tiles, cudaStream_t stream) {
  ts.n_kc = (ts.nKT + kTileCols - 1) / kTileCols;
  const unsigned grid = static_cast<unsigned>(tiles * ts.n_kc);
  return keep ? launch_pdl(tile_scales_kernel<true>, grid, kTileThreads, 0, stream, ts)
              : launch_pdl(tile_scales_kernel<false>, grid, kTileThreads, 0, stream, ts);
}

// ---------------------------------------------------------------------
// The fused gather through the scatter path.  One kernel builds the inverse
// of the row -> token map in a caller-provided workspace: every valid row r of
// token t takes slot atomicAdd(count[t], 1) of the token's bucket of
// kBucket rows, or, past kBucket routes, an entry of one overflow list.  The
// scatter kernel then reads and quantizes every token row once for the rows
// in its bucket (one warp per token) and once more per overflow entry.  The
// order of the rows in a bucket is arbitrary (atomics) and does not matter:
// every route of a token receives the same bytes.
constexpr int kBucket = MXFP4_SCATTER_MAX_TOP_K;  // rows per token bucket (one warp)

struct InvertParams {
  const int32_t* __restrict__ row_index;  // [R] token of every row
  int64_t total_rows;                     // R
  int64_t num_src_rows;                   // T
  int32_t* __restrict__ count;            // [T], zero on entry: routes of every token
  int32_t* __restrict__ ovf_n;            // [1], zero on entry: overflow entries
  int32_t* __restrict__ bucket;           // [T, kBucket] the first kBucket rows of every token
  int32_t* __restrict__ ovf_row;          // [R] rows past their token's kBucket-th
  int32_t* __restrict__ ovf_tok;          // [R] and their tokens
  int32_t* __restrict__ tok1;             // or NULL; else [padded rows], zero on entry: token + 1
                                          //   of every padded row with a valid index
  uint8_t* __restrict__ codes;            // rows with an index out of range are zeroed
  uint8_t* __restrict__ scales;           //   here: codes, and scale words unless tok1
  int64_t code_ld;
  const int32_t* __restrict__ offsets;
  const int32_t* __restrict__ padded;
  int32_t E;
  int32_t nKT;
  int32_t* status;
  int64_t code_rows;                      // zero codes only for bad rows below it
#ifdef MXFP4_DEBUG_BOUNDS
  DebugRanges dbg;  // kDbgCodes, kDbgScales, kDbgOffsets, kDbgPadded, kDbgRowIndex, kDbgStatus, kDbgWork
#endif
};

__global__ void __launch_bounds__(kInvertThreads) invert_bucket_kernel(const InvertParams q) {
  __shared__ int32_t s_off[kSmemSegs + 1];
  __shared__ int32_t s_pad[kSmemSegs + 1];
  pdl_wait();
  pdl_release();
  if (!MXFP4_IN_BOUNDS(q, kDbgPadded, q.padded, (q.E + 1) * 4) ||
      !MXFP4_IN_BOUNDS(q, kDbgOffsets, q.offsets, (q.E + 1) * 4) || __ldg(q.padded + q.E) < 0)
    return;  // rejected offsets: nothing is written (uniform over the block)
  const SegmentSearch seg(s_off, s_pad, q.offsets, q.padded, q.E,
                          static_cast<int>(q.total_rows));
  bool bad = false;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kInvertThreads;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kInvertThreads + threadIdx.x;
       r < q.total_rows; r += stride) {
    const int32_t* ip = q.row_index + r;
    const int32_t t = MXFP4_IN_BOUNDS(q, kDbgRowIndex, ip, 4) ? __ldg(ip) : -1;
    const bool valid = t >= 0 && t < q.num_src_rows;
    if (valid && MXFP4_IN_BOUNDS(q, kDbgWork, q.count + t, 4)) {
      const int32_t pos = atomicAdd(q.count + t, 1);
      if (pos < kBucket) {
        int32_t* const bp = q.bucket + static_cast<int64_t>(t) * kBucket + pos;
        if (MXFP4_IN_BOUNDS(q, kDbgWork, bp, 4)) *bp = static_cast<int32_t>(r);
      } else if (MXFP4_IN_BOUNDS(q, kDbgWork, q.ovf_n, 4)) {
        const int32_t j = atomicAdd(q.ovf_n, 1);  // < R: each row adds at most once
        if (MXFP4_IN_BOUNDS(q, kDbgWork, q.ovf_row + j, 4) &&
            MXFP4_IN_BOUNDS(q, kDbgWork, q.ovf_tok + j, 4)) {
          q.ovf_row[j] = static_cast<int32_t>(r);
          q.ovf_tok[j] = t;
        }
      }
    }
    if (valid && q.tok1 == nullptr) continue;
    const int prow = seg.padded_row(static_cast<int>(r));
    if (valid) {
      if (MXFP4_IN_BOUNDS(q, kDbgWork, q.tok1 + prow, 4)) q.tok1[prow] = t + 1;
      continue;
    }
    bad = true;
    uint8_t* cp = q.codes + r * q.code_ld;
    for (int64_t i = 0; r < q.code_rows && i < q.code_ld; i += 16)
      if (MXFP4_IN_BOUNDS(q, kDbgCodes, cp + i, 16))
        *reinterpret_cast<uint4*>(cp + i) = make_uint4(0u, 0u, 0u, 0u);
    if (q.tok1 != nullptr) continue;  // the tile kernel writes its zero scale words
    const int64_t base = scale_word_base(prow, q.nKT);
    for (int kt = 0; kt < q.nKT; ++kt) {
      uint8_t* wp = q.scales + base + static_cast<int64_t>(kt) * kChunkBytes;
      if (MXFP4_IN_BOUNDS(q, kDbgScales, wp, 4)) *reinterpret_cast<uint32_t*>(wp) = 0u;
    }
  }
  if (bad && q.status != nullptr && MXFP4_IN_BOUNDS(q, kDbgStatus, q.status, 4))
    atomicExch(q.status, MXFP4_EINDEX);
}

}  // namespace

int64_t scatter_workspace_ints(int64_t num_tokens, int64_t total_rows, int64_t E, int64_t K) {
  return gather_tok_ints(total_rows, E) + gather_stage_ints(num_tokens, K);
}

cudaError_t launch_quantize_grouped_scatter(const void* x, int64_t num_tokens, int64_t K,
                                            int64_t ldx, const int32_t* dest_rows, int32_t top_k,
                                            int64_t total_rows, const int32_t* offsets, int32_t E,
                                            int32_t* workspace, uint8_t* codes, uint8_t* scales,
                                            int32_t* scale_row_offsets, int32_t* status,
                                            int64_t bound_tiles, bool f16, cudaStream_t stream) {
  // staged: [tok1 PT][stage num_tokens x stage_ld(nKT)] (PT is a multiple of 128)
  const bool staged = workspace != nullptr && total_rows > 0 && E > 0 && K > 0;
  const int64_t PT = staged ? gather_tok_ints(total_rows, E) : 0;
  cudaError_t err = cudaSuccess;
  if (staged) {  // first, so that the kernels below follow one another directly
    err = cudaMemsetAsync(workspace, 0, static_cast<size_t>(PT) * 4, stream);
    if (err != cudaSuccess) return err;
  }
  err = launch_offsets(offsets, E, total_rows, scale_row_offsets, status, stream);
  if (err != cudaSuccess || E == 0 || K == 0) return err;
  const int32_t nKT = (static_cast<int32_t>(K / kBlock) + kTileBlocks - 1) / kTileBlocks;
  int32_t map_ctas = 0;
  if (staged) {
    // the row map (routes and pad rows, about 4 items per thread) runs in the
    // first CTAs of the scatter launch, beside the token warps
    const int64_t items = num_tokens * top_k > static_cast<int64_t>(E) * kTileRows
                              ? num_tokens * top_k
                              : static_cast<int64_t>(E) * kTileRows;
    const int64_t need = (items + 4 * kThreads - 1) / (4 * kThreads);
    map_ctas = static_cast<int32_t>(need < 1 ? 1 : (need < sm_count() ? need : sm_count()));
  }
  ScatterParams p{};
  p.x = static_cast<const uint8_t*>(x);
  p.ldx_bytes = ldx * 2;
  p.num_tokens = num_tokens;
  p.code_ld = K / 2;
  p.codes = codes;
  p.scales = scales;
  p.sK = static_cast<int32_t>(K / kBlock);
  p.nKT = nKT;
  p.stage = staged ? reinterpret_cast<uint32_t*>(workspace + PT) : nullptr;
  p.pad_ctas = staged ? 0 : E;
  p.map_ctas = map_ctas;
  p.tok1 = staged ? workspace : nullptr;
  p.offsets = offsets;
  p.padded = scale_row_offsets;
  p.E = E;
  p.status = status;
  p.dest_rows = dest_rows;
  p.top_k = top_k;
  p.total_rows = total_rows;
  p.code_rows = total_rows;
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(p.dbg, kDbgX, x, num_tokens > 0 ? ((num_tokens - 1) * ldx + K) * 2 : 0);
  debug_range(p.dbg, kDbgCodes, codes, total_rows * (K / 2));
  debug_range(p.dbg, kDbgScales, scales, bound_tiles * p.nKT * kChunkBytes);
  debug_range(p.dbg, kDbgOffsets, offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(p.dbg, kDbgPadded, scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(p.dbg, kDbgRowIndex, dest_rows, num_tokens * top_k * 4);
  debug_range(p.dbg, kDbgStatus, status, status ? 4 : 0);
  debug_range(p.dbg, kDbgWork, workspace, staged ? (PT + gather_stage_ints(num_tokens, K)) * 4 : 0);
#endif
  const int64_t grid =
      p.pad_ctas + p.map_ctas + (num_tokens + kScatterWarps - 1) / kScatterWarps;
  const bool v32 = vec32_ok(x, p.ldx_bytes);
  using Kernel = void (*)(const ScatterParams);
  static constexpr Kernel kKernels[2][2][2] = {
      {{quantize_scatter_kernel<false, false, false>, quantize_scatter_kernel<false, false, true>},
       {quantize_scatter_kernel<false, true, false>, quantize_scatter_kernel<false, true, true>}},
      {{quantize_scatter_kernel<true, false, false>, quantize_scatter_kernel<true, false, true>},
       {quantize_scatter_kernel<true, true, false>, quantize_scatter_kernel<true, true, true>}}};
  if (grid > 0) {
    err = launch_pdl(kKernels[v32][f16][staged], static_cast<unsigned>(grid), kThreads, 0, stream,
                     p);
    if (err != cudaSuccess) return err;
  }
  if (!staged || bound_tiles == 0) return cudaSuccess;
  TileScalesParams ts{};
  ts.tok1 = workspace;
  ts.stage = p.stage;
  ts.scales = scales;
  ts.padded = scale_row_offsets;
  ts.E = E;
  ts.nKT = nKT;
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(ts.dbg, kDbgScales, scales, bound_tiles * ts.nKT * kChunkBytes);
  debug_range(ts.dbg, kDbgPadded, scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(ts.dbg, kDbgRowIndex, workspace, PT * 4);
  debug_range(ts.dbg, kDbgWork, p.stage, gather_stage_ints(num_tokens, K) * 4);
#endif
  return launch_tile_scales(true, ts, bound_tiles, stream);
}

// Workspace of the gather through the scatter path, in int32:
//   [count T][ovf_n 1][tok1 PT, staged only]  cleared by one memset
//   [bucket T x kBucket][ovf_row R][ovf_tok R]
//   [stage T x stage_ld(nKT), staged only]    from the next 16-byte boundary
int64_t gather_workspace_ints(int64_t num_src_rows, int64_t total_rows) {
  return num_src_rows * (1 + kBucket) + 1 + 2 * total_rows;
}

int64_t gather_tok_ints(int64_t total_rows, int64_t E) {
  return (total_rows + 127 * E) / kTileRows * kTileRows;
}

int64_t gather_stage_ints(int64_t num_src_rows, int64_t K) {
  return num_src_rows * stage_ld(static_cast<int>((K / kBlock + kTileBlocks - 1) / kTileBlocks));
}

namespace {

// The gather through the scatter path.  borrowed: the workspace is the tail
// of `codes` from row code_rows on; it is cleared by a kernel (only for valid
// offsets) and those rows' codes are written last by gather_row_codes_kernel.
cudaError_t gather_ws_impl(const void* x, int64_t num_src_rows, int64_t K, int64_t ldx,
                           const int32_t* row_index, int64_t total_rows, const int32_t* offsets,
                           int32_t E, int32_t* workspace, bool staged, bool borrowed,
                           int64_t code_rows, uint8_t* codes, uint8_t* scales,
                           int32_t* scale_row_offsets, int32_t* status, int64_t bound_tiles,
                           bool f16, cudaStream_t stream) {
  const int64_t T = num_src_rows;
  const int64_t R = total_rows;
  const int64_t PT = staged ? gather_tok_ints(R, E) : 0;
  // no rows: every segment is empty and nothing but the offsets is written
  // (the caller need not pass a workspace then)
  const bool work = E > 0 && K > 0 && R > 0;
  cudaError_t err = cudaSuccess;
  if (work && !borrowed) {  // first, so that the kernels below follow one another directly
    err = cudaMemsetAsync(workspace, 0, static_cast<size_t>(T + 1 + PT) * 4, stream);
    if (err != cudaSuccess) return err;
  }
  err = launch_offsets(offsets, E, total_rows, scale_row_offsets, status, stream);
  if (err != cudaSuccess || !work) return err;
  if (borrowed) {  // T + 1 + PT ints, rounded up to whole uint4 (the map region is larger)
    const int64_t n16 = (T + 1 + PT + 3) / 4;
    const int64_t need = (n16 + kThreads - 1) / kThreads;
    const unsigned ctas = static_cast<unsigned>(need < sm_count() ? need : sm_count());
    err = launch_pdl(clear_words_kernel, ctas, kThreads, 0, stream, scale_row_offsets, E,
                     reinterpret_cast<uint4*>(workspace), n16);
    if (err != cudaSuccess) return err;
  }
  InvertParams q{};
  q.row_index = row_index;
  q.total_rows = R;
  q.num_src_rows = T;
  q.count = workspace;
  q.ovf_n = workspace + T;
  q.tok1 = staged ? workspace + T + 1 : nullptr;
  q.bucket = workspace + T + 1 + PT;
  q.ovf_row = q.bucket + T * kBucket;
  q.ovf_tok = q.ovf_row + R;
  q.codes = codes;
  q.scales = scales;
  q.code_ld = K / 2;
  q.offsets = offsets;
  q.padded = scale_row_offsets;
  q.E = E;
  q.nKT = (static_cast<int32_t>(K / kBlock) + kTileBlocks - 1) / kTileBlocks;
  q.status = status;
  q.code_rows = code_rows;
  const int64_t map_ints = (gather_workspace_ints(T, R) + PT + 3) & ~int64_t{3};
  const int64_t ws_bytes = (map_ints + (staged ? gather_stage_ints(T, K) : 0)) * 4;
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(q.dbg, kDbgCodes, codes, R * (K / 2));
  debug_range(q.dbg, kDbgScales, scales, bound_tiles * q.nKT * kChunkBytes);
  debug_range(q.dbg, kDbgOffsets, offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(q.dbg, kDbgPadded, scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(q.dbg, kDbgRowIndex, row_index, R * 4);
  debug_range(q.dbg, kDbgStatus, status, status ? 4 : 0);
  debug_range(q.dbg, kDbgWork, workspace, ws_bytes);
#endif
  const int64_t row_ctas_max = static_cast<int64_t>(sm_count()) * 8;
  const int64_t need = (R + kInvertThreads - 1) / kInvertThreads;
  const unsigned row_ctas =
      static_cast<unsigned>(need < 1 ? 1 : (need < row_ctas_max ? need : row_ctas_max));
  if ((err = launch_pdl(invert_bucket_kernel, row_ctas, kInvertThreads, 0, stream, q)) !=
      cudaSuccess)
    return err;
  ScatterParams p{};
  p.x = static_cast<const uint8_t*>(x);
  p.ldx_bytes = ldx * 2;
  p.num_tokens = T;
  p.dest_rows = q.bucket;
  p.count = q.count;
  p.ovf_n = q.ovf_n;
  p.ovf_row = q.ovf_row;
  p.ovf_tok = q.ovf_tok;
  p.top_k = 0;
  p.E = E;
  p.total_rows = R;
  p.code_ld = K / 2;
  p.codes = codes;
  p.scales = scales;
  p.offsets = offsets;
  p.padded = scale_row_offsets;
  p.status = status;
  p.stage = staged ? reinterpret_cast<uint32_t*>(workspace + map_ints) : nullptr;
  p.pad_ctas = staged ? 0 : E;
  p.sK = static_cast<int32_t>(K / kBlock);
  p.nKT = q.nKT;
  p.code_rows = code_rows;
  // one warp per token, then up to one CTA per SM of warps for the overflow
  // list (the token CTAs' spare warps walk it too)
  const int64_t token_ctas = (T + kScatterWarps - 1) / kScatterWarps;
  const int64_t ovf_need = (R + kScatterWarps - 1) / kScatterWarps;
  const int64_t ovf_ctas = ovf_need < sm_count() ? ovf_need : sm_count();
  p.n_ovf_warps = static_cast<int32_t>((token_ctas + ovf_ctas) * kScatterWarps - T);
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(p.dbg, kDbgX, x, T > 0 ? ((T - 1) * ldx + K) * 2 : 0);
  debug_range(p.dbg, kDbgCodes, codes, R * (K / 2));
  debug_range(p.dbg, kDbgScales, scales, bound_tiles * p.nKT * kChunkBytes);
  debug_range(p.dbg, kDbgOffsets, offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(p.dbg, kDbgPadded, scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(p.dbg, kDbgRowIndex, q.bucket, (T * kBucket + R) * 4);  // buckets + ovf_row
  debug_range(p.dbg, kDbgStatus, status, status ? 4 : 0);
  debug_range(p.dbg, kDbgWork, workspace, ws_bytes);
#else
  (void)ws_bytes;
#endif
  const int64_t grid = p.pad_ctas + token_ctas + ovf_ctas;
  const bool v32 = vec32_ok(x, p.ldx_bytes);
  using Kernel = void (*)(const ScatterParams);
  static constexpr Kernel kKernels[2][2][2] = {
      {{quantize_scatter_kernel<false, false, false>, quantize_scatter_kernel<false, false, true>},
       {quantize_scatter_kernel<false, true, false>, quantize_scatter_kernel<false, true, true>}},
      {{quantize_scatter_kernel<true, false, false>, quantize_scatter_kernel<true, false, true>},
       {quantize_scatter_kernel<true, true, false>, quantize_scatter_kernel<true, true, true>}}};
  err = launch_pdl(kKernels[v32][f16][staged], static_cast<unsigned>(grid), kThreads, 0, stream,
                   p);
  if (err != cudaSuccess || !staged || bound_tiles == 0) return err;
  TileScalesParams ts{};
  ts.tok1 = q.tok1;
  ts.stage = p.stage;
  ts.scales = scales;
  ts.padded = scale_row_offsets;
  ts.E = E;
  ts.nKT = q.nKT;
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(ts.dbg, kDbgScales, scales, bound_tiles * ts.nKT * kChunkBytes);
  debug_range(ts.dbg, kDbgPadded, scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(ts.dbg, kDbgRowIndex, q.tok1, PT * 4);
  debug_range(ts.dbg, kDbgWork, p.stage, T * stage_ld(ts.nKT) * 4);
#endif
  err = launch_tile_scales(false, ts, bound_tiles, stream);
  if (err != cudaSuccess || code_rows >= R) return err;
  RowCodesParams rc{};
  rc.x = static_cast<const uint8_t*>(x);
  rc.ldx_bytes = ldx * 2;
  rc.num_src_rows = T;
  rc.row_index = row_index;
  rc.r0 = code_rows;
  rc.total_rows = R;
  rc.codes = codes;
  rc.code_ld = K / 2;
  rc.padded = scale_row_offsets;
  rc.E = E;
  rc.sK = static_cast<int32_t>(K / kBlock);
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(rc.dbg, kDbgX, x, T > 0 ? ((T - 1) * ldx + K) * 2 : 0);
  debug_range(rc.dbg, kDbgCodes, codes, R * (K / 2));
  debug_range(rc.dbg, kDbgPadded, scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(rc.dbg, kDbgRowIndex, row_index, R * 4);
#endif
  const int64_t n_pass = (K / kBlock + 15) / 16;
  const int64_t warps = (R - code_rows) * ((n_pass + kRowGroup - 1) / kRowGroup);
  const auto row_kernel = f16 ? (v32 ? gather_row_codes_kernel<true, true>
                                     : gather_row_codes_kernel<false, true>)
                              : (v32 ? gather_row_codes_kernel<true, false>
                                     : gather_row_codes_kernel<false, false>);
  return launch_pdl(row_kernel, static_cast<unsigned>((warps + kScatterWarps - 1) / kScatterWarps),
                    kThreads, 0, stream, rc);
}

}  // namespace

cudaError_t launch_quantize_grouped_gather_ws(const void* x, int64_t num_src_rows, int64_t K,
                                              int64_t ldx, const int32_t* row_index,
                                              int64_t total_rows, const int32_t* offsets,
                                              int32_t E, int32_t* workspace, bool staged,
                                              uint8_t* codes, uint8_t* scales,
                                              int32_t* scale_row_offsets, int32_t* status,
                                              int64_t bound_tiles, bool f16, cudaStream_t stream) {
  return gather_ws_impl(x, num_src_rows, K, ldx, row_index, total_rows, offsets, E, workspace,
                        staged, false, total_rows, codes, scales, scale_row_offsets, status,
                        bound_tiles, f16, stream);
}

int64_t gather_borrow_rows(int64_t num_src_rows, int64_t total_rows, int64_t E, int64_t K) {
  if (K <= 0 || total_rows <= 0) return -1;
  const int64_t map_ints =
      (gather_workspace_ints(num_src_rows, total_rows) + gather_tok_ints(total_rows, E) + 3) &
      ~int64_t{3};
  const int64_t bytes = (map_ints + gather_stage_ints(num_src_rows, K)) * 4;
  const int64_t rows = (bytes + K / 2 - 1) / (K / 2);
  return rows * 4 <= total_rows ? rows : -1;  // the codes of at most a quarter of the rows
}

cudaError_t launch_quantize_grouped_gather_borrowed(const void* x, int64_t num_src_rows,
                                                    int64_t K, int64_t ldx,
                                                    const int32_t* row_index, int64_t total_rows,
                                                    const int32_t* offsets, int32_t E,
                                                    uint8_t* codes, uint8_t* scales,
                                                    int32_t* scale_row_offsets, int32_t* status,
                                                    int64_t bound_tiles, bool f16,
                                                    cudaStream_t stream) {
  const int64_t tail = gather_borrow_rows(num_src_rows, total_rows, E, K);
  if (tail < 0) return cudaErrorInvalidValue;
  const int64_t r0 = total_rows - tail;
  int32_t* const workspace = reinterpret_cast<int32_t*>(codes + r0 * (K / 2));
  return gather_ws_impl(x, num_src_rows, K, ldx, row_index, total_rows, offsets, E, workspace,
                        true, true, r0, codes, scales, scale_row_offsets, status, bound_tiles,
                        f16, stream);
}

// NVFP4 experts quant with the dispatch as a scatter.  Workspace (staged):
// [tok1: PT int32][stage: PT rows x stage_ld(nKT) words], PT padded rows.
int64_t nvfp4_scatter_workspace_ints(int64_t total_rows, int64_t E, int64_t K) {
  const int32_t nKT = static_cast<int32_t>((K / 16 + kTileBlocks - 1) / kTileBlocks);
  return gather_tok_ints(total_rows, E) * (1 + stage_ld(nKT));
}

cudaError_t launch_quantize_nvfp4_grouped_scatter(const void* x, int64_t num_tokens, int64_t K,
                                                  int64_t ldx, const int32_t* dest_rows,
                                                  int32_t top_k, int64_t total_rows,
                                                  const int32_t* offsets, int32_t E,
                                                  const float* global_scales, int32_t* workspace,
                                                  uint8_t* codes, uint8_t* scales,
                                                  int32_t* scale_row_offsets, int32_t* status,
                                                  int64_t bound_tiles, bool f16,
                                                  cudaStream_t stream) {
  const bool staged = workspace != nullptr && total_rows > 0 && E > 0 && K > 0;
  const int64_t PT = staged ? gather_tok_ints(total_rows, E) : 0;
  cudaError_t err = cudaSuccess;
  if (staged) {  // first, so that the kernels below follow one another directly
    err = cudaMemsetAsync(workspace, 0, static_cast<size_t>(PT) * 4, stream);
    if (err != cudaSuccess) return err;
  }
  err = launch_offsets(offsets, E, total_rows, scale_row_offsets, status, stream);
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
  p.sK = static_cast<int32_t>(K / 16);
  p.nKT = (p.sK + kTileBlocks - 1) / kTileBlocks;
  p.pad_ctas = staged ? 0 : E;
  if (staged) {
    // the map CTAs write the pad rows only (the token warps the routed rows)
    const int64_t items = static_cast<int64_t>(E) * kTileRows;
    const int64_t need = (items + 4 * kThreads - 1) / (4 * kThreads);
    p.map_ctas = static_cast<int32_t>(need < 1 ? 1 : (need < sm_count() ? need : sm_count()));
    p.tok1 = workspace;
    p.stage = reinterpret_cast<uint8_t*>(workspace + PT);
  }
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(p.dbg, kDbgX, x, num_tokens > 0 ? ((num_tokens - 1) * ldx + K) * 2 : 0);
  debug_range(p.dbg, kDbgCodes, codes, total_rows * (K / 2));
  debug_range(p.dbg, kDbgScales, scales, bound_tiles * p.nKT * kChunkBytes);
  debug_range(p.dbg, kDbgOffsets, offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(p.dbg, kDbgPadded, scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(p.dbg, kDbgRowIndex, dest_rows, num_tokens * top_k * 4);
  debug_range(p.dbg, kDbgStatus, status, status ? 4 : 0);
  debug_range(p.dbg, kDbgWork, workspace, staged ? PT * (1 + stage_ld(p.nKT)) * 4 : 0);
  debug_range(p.dbg_g, 0, global_scales, static_cast<int64_t>(E) * 4);
#endif
  const int64_t grid =
      p.pad_ctas + p.map_ctas + (num_tokens + kScatterWarps - 1) / kScatterWarps;
  const bool v32 = vec32_ok(x, p.ldx_bytes);
  using Kernel = void (*)(const Nvfp4ScatterParams);
  static constexpr Kernel kKernels[2][2][2] = {
      {{nvfp4_scatter_kernel<false, false, false>, nvfp4_scatter_kernel<false, false, true>},
       {nvfp4_scatter_kernel<false, true, false>, nvfp4_scatter_kernel<false, true, true>}},
      {{nvfp4_scatter_kernel<true, false, false>, nvfp4_scatter_kernel<true, false, true>},
       {nvfp4_scatter_kernel<true, true, false>, nvfp4_scatter_kernel<true, true, true>}}};
  if (grid > 0) {
    err = launch_pdl(kKernels[v32][f16][staged], static_cast<unsigned>(grid), kThreads, 0, stream,
                     p);
    if (err != cudaSuccess) return err;
  }
  if (!staged || bound_tiles == 0) return cudaSuccess;
  TileScalesParams ts{};
  ts.tok1 = workspace;
  ts.stage = reinterpret_cast<const uint32_t*>(p.stage);
  ts.scales = scales;
  ts.padded = scale_row_offsets;
  ts.E = E;
  ts.nKT = p.nKT;
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(ts.dbg, kDbgScales, scales, bound_tiles * ts.nKT * kChunkBytes);
  debug_range(ts.dbg, kDbgPadded, scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(ts.dbg, kDbgRowIndex, workspace, PT * 4);
  debug_range(ts.dbg, kDbgWork, p.stage, PT * stage_ld(ts.nKT) * 4);
#endif
  return launch_tile_scales(true, ts, bound_tiles, stream);
}

#ifdef MXFP4_DEBUG_BOUNDS
unsigned int debug_violations_dispatch() {
  unsigned int v = 0, zero = 0;
  cudaMemcpyFromSymbol(&v, g_debug_violations, sizeof v);
  cudaMemcpyToSymbol(g_debug_violations, &zero, sizeof zero);
  return v;
}
#endif

}  // namespace mxfp4
