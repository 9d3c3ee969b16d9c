// route.cu — the MoE dispatch permutation from the router's expert ids, for
// sm_103a: the expert-sorted row order the experts quant consumes (vLLM PR
// #43557 page, "Implementation breakdown" item 3: the routed activations,
// sorted by expert), as the offsets, token -> rows and row -> token maps the
// grouped, scatter and gather calls take.
//
// Entry i = t * top_k + j of the ids is route j of token t.  Rows are the
// entries with an expert in [0, E), in order of expert and, within an expert,
// of entry index (a stable counting sort); -1 marks a route that is not
// dispatched, any other id outside [0, E) is not dispatched either and is
// reported.  Three kernels, each a fixed function of the previous one's
// output, with no waiting between CTAs (with no entries at all, a memset and
// route_expert_scan_kernel write the zero offsets and the status instead):
//   1. route_count_kernel: one CTA per chunk of kRouteChunk entries counts
//      its entries per expert (shared-memory atomics; the order of the adds
//      does not matter) and flags an invalid id;
//   2. route_chunk_scan_kernel: per expert, the exclusive prefix of those
//      counts over the chunks, and the expert's total; the CTA that finishes
//      last (an atomic ticket, taken after its writes are fenced) then scans
//      the totals over the experts (the offsets) and writes the status word;
//   3. route_place_kernel: one warp per chunk walks its entries in order,
//      32 at a time; lanes with the same expert find one another with
//      __match_any_sync and take consecutive rows in lane order.
#include <cstdint>

#include <cuda_runtime.h>

#include "mxfp4_device.cuh"
#include "mxfp4_internal.h"
#include "../../include/mxfp4.h"

namespace mxfp4 {
namespace {

constexpr int kRouteChunk = 256;  // entries per count CTA and per placing warp
constexpr int kCountThreads = 256;
constexpr int kScanThreads = 1024;

struct RouteParams {
  const int32_t* __restrict__ ids;  // [n]
  int32_t n;                        // entries = num_tokens * top_k
  int32_t top_k;
  int32_t E;
  int32_t n_ch;                     // chunks of kRouteChunk entries
  int32_t* __restrict__ counts;     // workspace: [n_ch, E] counts, then row bases
  int32_t* __restrict__ bad;        // workspace: [n_ch] chunk has an invalid id
  unsigned int* ticket;             // workspace: CTAs of the chunk scan done
  int32_t* __restrict__ offsets;    // [E+1]
  int32_t* __restrict__ dest;       // [n]
  int32_t* __restrict__ row_index;  // [rows] or NULL
  int32_t* status;                  // or NULL
#ifdef MXFP4_DEBUG_BOUNDS
  DebugRanges dbg;
#endif
};

enum : int {
  kDbgIds = 0, kDbgCounts, kDbgBad, kDbgOffsets, kDbgDest, kDbgRowIndex, kDbgStatus, kDbgTicket
};

__global__ void __launch_bounds__(kCountThreads) route_count_kernel(const RouteParams p) {
  extern __shared__ int32_t s_hist[];
  __shared__ int s_bad;
  pdl_wait();
  pdl_release();
  for (int e = threadIdx.x; e < p.E; e += kCountThreads) s_hist[e] = 0;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kRouteChunk;
  int bad = 0;
  for (int i = threadIdx.x; i < kRouteChunk; i += kCountThreads) {
    const int64_t id = base + i;
    if (id < p.n && MXFP4_IN_BOUNDS(p, kDbgIds, p.ids + id, 4)) {
      const int32_t e = __ldg(p.ids + id);
      if (e >= 0 && e < p.E) atomicAdd(&s_hist[e], 1);
      else if (e != -1) bad = 1;
    }
  }
  if (bad) atomicOr(&s_bad, 1);
  __syncthreads();
  int32_t* const row = p.counts + static_cast<int64_t>(blockIdx.x) * p.E;
  for (int e = threadIdx.x; e < p.E; e += kCountThreads)
    if (MXFP4_IN_BOUNDS(p, kDbgCounts, row + e, 4)) row[e] = s_hist[e];
  if (threadIdx.x == 0 && MXFP4_IN_BOUNDS(p, kDbgBad, p.bad + blockIdx.x, 4))
    p.bad[blockIdx.x] = s_bad;
  // the chunk scan, a later launch, counts its finished CTAs from zero
  if (blockIdx.x == 0 && threadIdx.x == 0 && MXFP4_IN_BOUNDS(p, kDbgTicket, p.ticket, 4))
    *p.ticket = 0u;
}

// offsets[e] holds expert e's total: replace every total by the exclusive
// scan over the experts, write offsets[E] and the status word (MXFP4_EINDEX
// when some chunk saw an invalid id).  Run by one CTA of kScanThreads; the
// totals are read from the L2 (other CTAs wrote them).
__device__ void scan_expert_totals(const RouteParams& p) {
  __shared__ int32_t s_warp[kScanThreads / 32];
  __shared__ int32_t s_carry;
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_carry = 0;
    s_bad = 0;
  }
  __syncthreads();
  int bad = 0;
  for (int c = tid; c < p.n_ch; c += kScanThreads)
    if (MXFP4_IN_BOUNDS(p, kDbgBad, p.bad + c, 4) && __ldcg(p.bad + c)) bad = 1;
  if (bad) atomicOr(&s_bad, 1);
  __syncthreads();
  for (int base = 0; base < p.E; base += kScanThreads) {
    const int e = base + tid;
    const int32_t v =
        (e < p.E && MXFP4_IN_BOUNDS(p, kDbgOffsets, p.offsets + e, 4)) ? __ldcg(p.offsets + e) : 0;
    int32_t inc = v;  // inclusive warp scan
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t t = __shfl_up_sync(0xFFFFFFFFu, inc, d);
      if (lane >= d) inc += t;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
      int32_t w = s_warp[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int32_t t = __shfl_up_sync(0xFFFFFFFFu, w, d);
        if (lane >= d) w += t;
      }
      s_warp[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int32_t before = s_carry + (warp > 0 ? s_warp[warp - 1] : 0) + inc - v;
    if (e < p.E && MXFP4_IN_BOUNDS(p, kDbgOffsets, p.offsets + e, 4)) p.offsets[e] = before;
    __syncthreads();
    if (tid == 0) s_carry += s_warp[kScanThreads / 32 - 1];
    __syncthreads();
  }
  if (tid == 0) {
    if (MXFP4_IN_BOUNDS(p, kDbgOffsets, p.offsets + p.E, 4)) p.offsets[p.E] = s_carry;
    if (p.status != nullptr && MXFP4_IN_BOUNDS(p, kDbgStatus, p.status, 4))
      *p.status = s_bad ? MXFP4_EINDEX : MXFP4_OK;
  }
}

// One CTA per 32 experts: thread (s, lane) sums its expert's counts over a
// slice of the chunks; warp 0 turns the 32 slice sums of every expert into
// exclusive prefixes (and the expert's total, left in offsets[e]); each
// thread then rewrites its slice's counts as running prefixes.
__global__ void __launch_bounds__(kScanThreads, 1) route_chunk_scan_kernel(const RouteParams p) {
  __shared__ int32_t s_part[32][32];
  pdl_wait();
  pdl_release();
  const int lane = threadIdx.x & 31;
  const int s = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + lane;
  const int per = (p.n_ch + 31) / 32;
  const int c0 = s * per;
  const int c1 = min(p.n_ch, c0 + per);
  // the slice's counts stay in registers between the sum and the rewrite
  // when it has at most kHeld chunks (every load in flight at once)
  constexpr int kHeld = 16;
  int32_t held[kHeld];
  int32_t sum = 0;
  if (e < p.E) {
    if (c1 - c0 <= kHeld) {
#pragma unroll
      for (int k = 0; k < kHeld; ++k) {
        const int32_t* cp = p.counts + static_cast<int64_t>(c0 + k) * p.E + e;
        held[k] = (c0 + k < c1 && MXFP4_IN_BOUNDS(p, kDbgCounts, cp, 4)) ? *cp : 0;
      }
#pragma unroll
      for (int k = 0; k < kHeld; ++k) sum += held[k];
    } else {
      for (int c = c0; c < c1; ++c) {
        const int32_t* cp = p.counts + static_cast<int64_t>(c) * p.E + e;
        if (MXFP4_IN_BOUNDS(p, kDbgCounts, cp, 4)) sum += *cp;
      }
    }
  }
  s_part[s][lane] = sum;
  __syncthreads();
  if (s == 0) {
    int32_t run = 0;
    for (int k = 0; k < 32; ++k) {
      const int32_t v = s_part[k][lane];
      s_part[k][lane] = run;
      run += v;
    }
    if (e < p.E && MXFP4_IN_BOUNDS(p, kDbgOffsets, p.offsets + e, 4)) p.offsets[e] = run;
  }
  __syncthreads();
  int32_t run = s_part[s][lane];
  if (e < p.E) {
    if (c1 - c0 <= kHeld) {
#pragma unroll
      for (int k = 0; k < kHeld; ++k) {
        int32_t* cp = p.counts + static_cast<int64_t>(c0 + k) * p.E + e;
        if (c0 + k < c1 && MXFP4_IN_BOUNDS(p, kDbgCounts, cp, 4)) *cp = run;
        run += held[k];
      }
    } else {
      for (int c = c0; c < c1; ++c) {
        int32_t* cp = p.counts + static_cast<int64_t>(c) * p.E + e;
        if (MXFP4_IN_BOUNDS(p, kDbgCounts, cp, 4)) {
          const int32_t v = *cp;
          *cp = run;
          run += v;
        }
      }
    }
  }
  // the last CTA to finish scans the totals of all of them
  __shared__ bool s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0)
    s_last = MXFP4_IN_BOUNDS(p, kDbgTicket, p.ticket, 4) &&
             atomicAdd(p.ticket, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  scan_expert_totals(p);
}

// With no entries: one CTA scans the (zero) totals and writes the status.
__global__ void __launch_bounds__(kScanThreads) route_expert_scan_kernel(const RouteParams p) {
  pdl_wait();
  pdl_release();
  scan_expert_totals(p);
}

// One warp per chunk, its entries in order, 32 a step.  The row of an entry
// of expert e is offsets[e] + (e's entries in earlier chunks) + (e's entries
// earlier in this chunk): the first two terms are loaded per entry, all of
// them in flight together; the third is a running count per expert in shared
// memory, where at each step the lanes holding one expert take consecutive
// rows in lane order and the lowest of them advances the count.
__global__ void __launch_bounds__(32) route_place_kernel(const RouteParams p) {
  extern __shared__ int32_t s_run[];
  constexpr int kSteps = kRouteChunk / 32;
  pdl_wait();
  pdl_release();
  const int lane = threadIdx.x;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kRouteChunk;
  const int32_t* const brow = p.counts + static_cast<int64_t>(blockIdx.x) * p.E;
  for (int e = lane; e < p.E; e += 32) s_run[e] = 0;
  int32_t id_e[kSteps];
#pragma unroll
  for (int k = 0; k < kSteps; ++k) {
    const int64_t id = base + k * 32 + lane;
    id_e[k] = (id < p.n && MXFP4_IN_BOUNDS(p, kDbgIds, p.ids + id, 4)) ? __ldg(p.ids + id) : -1;
  }
  int32_t first[kSteps];  // offsets[e] + e's entries in earlier chunks
#pragma unroll
  for (int k = 0; k < kSteps; ++k) {
    const int32_t e = id_e[k];
    first[k] = 0;
    if (e >= 0 && e < p.E && MXFP4_IN_BOUNDS(p, kDbgCounts, brow + e, 4) &&
        MXFP4_IN_BOUNDS(p, kDbgOffsets, p.offsets + e, 4))
      first[k] = brow[e] + p.offsets[e];
  }
  __syncwarp();
  uint32_t lt;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(lt));
  // token t and route j of this lane's entry, advanced by 32 entries a step
  // (32 = adv_t * top_k + adv_j) instead of a division per entry
  const int32_t id0 = static_cast<int32_t>(base) + lane;
  int32_t t = id0 / p.top_k;
  int32_t j = id0 - t * p.top_k;
  const int32_t adv_t = 32 / p.top_k;
  const int32_t adv_j = 32 - adv_t * p.top_k;
#pragma unroll
  for (int k = 0; k < kSteps; ++k) {
    const int64_t id = base + k * 32 + lane;
    const int32_t e = id_e[k];
    const bool valid = id < p.n && e >= 0 && e < p.E;
    // lanes without a valid expert get keys of their own
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, valid ? e : -1 - lane);
    const int rank = __popc(peers & lt);
    if (valid) {
      const int32_t row = first[k] + s_run[e] + rank;
      if (MXFP4_IN_BOUNDS(p, kDbgDest, p.dest + id, 4)) p.dest[id] = row;
      if (p.row_index != nullptr && MXFP4_IN_BOUNDS(p, kDbgRowIndex, p.row_index + row, 4))
        p.row_index[row] = t;
    } else if (id < p.n && MXFP4_IN_BOUNDS(p, kDbgDest, p.dest + id, 4)) {
      p.dest[id] = -1;
    }
    __syncwarp();
    if (valid && rank == 0) s_run[e] += __popc(peers);
    __syncwarp();
    t += adv_t;
    j += adv_j;
    if (j >= p.top_k) {
      j -= p.top_k;
      ++t;
    }
  }
}

}  // namespace

int64_t route_workspace_ints(int64_t n, int64_t E) {
  const int64_t n_ch = (n + kRouteChunk - 1) / kRouteChunk;
  return n_ch * (E + 1) + 4;  // counts, chunk flags, the ticket (padded to 16 bytes)
}

cudaError_t launch_moe_route(const int32_t* ids, int64_t num_tokens, int32_t top_k, int32_t E,
                             int32_t* workspace, int32_t* offsets, int32_t* dest,
                             int32_t* row_index, int32_t* status, cudaStream_t stream) {
  RouteParams p{};
  const int64_t n = num_tokens * top_k;
  p.ids = ids;
  p.n = static_cast<int32_t>(n);
  p.top_k = top_k;
  p.E = E;
  p.n_ch = static_cast<int32_t>((n + kRouteChunk - 1) / kRouteChunk);
  p.counts = workspace;
  p.bad = workspace + static_cast<int64_t>(p.n_ch) * E;
  p.ticket = reinterpret_cast<unsigned int*>(p.bad + p.n_ch);
  p.offsets = offsets;
  p.dest = dest;
  p.row_index = row_index;
  p.status = status;
#ifdef MXFP4_DEBUG_BOUNDS
  debug_range(p.dbg, kDbgIds, ids, n * 4);
  debug_range(p.dbg, kDbgCounts, workspace, static_cast<int64_t>(p.n_ch) * E * 4);
  debug_range(p.dbg, kDbgBad, p.bad, static_cast<int64_t>(p.n_ch) * 4);
  debug_range(p.dbg, kDbgOffsets, offsets, (static_cast<int64_t>(E) + 1) * 4);
  debug_range(p.dbg, kDbgDest, dest, n * 4);
  debug_range(p.dbg, kDbgRowIndex, row_index, row_index ? n * 4 : 0);
  debug_range(p.dbg, kDbgStatus, status, status ? 4 : 0);
  debug_range(p.dbg, kDbgTicket, p.ticket, 4);
#endif
  const size_t smem = static_cast<size_t>(E) * 4;
  cudaError_t err = cudaSuccess;
  if (p.n_ch > 0) {
    err = launch_pdl(route_count_kernel, static_cast<unsigned>(p.n_ch), kCountThreads, smem,
                     stream, p);
    if (err != cudaSuccess) return err;
    err = launch_pdl(route_chunk_scan_kernel, static_cast<unsigned>((E + 31) / 32),
                     kScanThreads, 0, stream, p);
    if (err != cudaSuccess) return err;
    return launch_pdl(route_place_kernel, static_cast<unsigned>(p.n_ch), 32, smem, stream, p);
  }
  // no entries: every expert's total is 0
  err = cudaMemsetAsync(offsets, 0, static_cast<size_t>(E) * 4, stream);
  if (err != cudaSuccess) return err;
  return launch_pdl(route_expert_scan_kernel, 1, kScanThreads, 0, stream, p);
}

#ifdef MXFP4_DEBUG_BOUNDS
unsigned int debug_violations_route() {
  unsigned int v = 0, zero = 0;
  cudaMemcpyFromSymbol(&v, g_debug_violations, sizeof v);
  cudaMemcpyToSymbol(g_debug_violations, &zero, sizeof zero);
  return v;
}
#endif

}  // namespace mxfp4
