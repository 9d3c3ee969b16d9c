// mxfp4_api.cu — the extern "C" entry points of libmxfp4_gb300.so.
//
// Each entry point validates its arguments on the host (no device access,
// no allocation, no synchronisation), then enqueues the kernels on the
// caller's stream.  See include/mxfp4.h for the contract of every call.
#include <climits>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "mxfp4_internal.h"
#include "../../include/mxfp4.h"
#ifdef MXFP4_DEBUG_BOUNDS
#include "../../include/mxfp4_debug.h"
#endif

namespace mxfp4 {

int sm_count() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
    cached[dev] = n;
  }
  return cached[dev];
}

// Fixed scratch of mxfp4_quantize_grouped_gather_noalloc: the inverse-map
// workspace of the gather-through-scatter path, for callers that cannot
// allocate.  Host code only ever uses its device address, looked up with the
// device current.
static __device__ __align__(256) int32_t g_noalloc_scratch[MXFP4_NOALLOC_SCRATCH_BYTES / 4];

// The process-unique id of the calling thread's current context (the
// driver's cuCtxGetCurrent and cuCtxGetId, reached through the runtime's
// driver entry points so that the library does not link libcuda), or 0 when
// there is none or the entry points are unavailable.
unsigned long long current_context_id() {
  using GetCurrent = int (*)(void**);
  using GetId = int (*)(void*, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  void* ctx = nullptr;
  if (get_current(&ctx) != 0 || ctx == nullptr) return 0;
  unsigned long long id = 0;
  return get_id(ctx, &id) == 0 ? id : 0;
}

// Device address of the scratch array in the current context.  The address
// is looked up on a device's first call and again whenever the current
// context is not the one it was looked up in (a cudaDeviceReset destroys the
// primary context, and the array then lives at a new address in the next
// one); context ids are never reused within a process.  Without a context id
// the address is looked up on every call.
int32_t* noalloc_scratch() {
  static std::mutex mu;
  static int32_t* cached[64] = {nullptr};
  static unsigned long long cached_ctx[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long id = current_context_id();
  if (id == 0 || cached[dev] == nullptr || cached_ctx[dev] != id) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<int32_t*>(ptr);
    // the lookup made the device's context current if none was
    cached_ctx[dev] = id != 0 ? id : current_context_id();
  }
  return cached[dev];
}

}  // namespace mxfp4

namespace {

constexpr int64_t kMaxGrid = INT_MAX / 2;  // tile counts stay far from int overflow

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
};

Range range_of(const void* p, int64_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Range{a, a + static_cast<uintptr_t>(bytes > 0 ? bytes : 0)};
}

bool overlap(Range a, Range b) {
  if (a.lo == a.hi || b.lo == b.hi) return false;
  return a.lo < b.hi && b.lo < a.hi;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? MXFP4_OK : MXFP4_ECUDA; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int64_t padded_scale_cols(int64_t K) { return ceil_div(K / 32, 4) * 4; }

// Byte count of `rows` rows of `cols` scale bytes for a size query, or 0 when
// it does not fit in int64 (no call accepts such sizes).
size_t rows_times_cols(int64_t rows, int64_t cols) {
  int64_t r = 0;
  return __builtin_mul_overflow(rows, cols, &r) ? 0 : static_cast<size_t>(r);
}

// Row counts above this are rejected by every call; the size queries return
// 0 for them instead of wrapping around.
constexpr int64_t kMaxRows = INT64_MAX / 4;

}  // namespace

extern "C" {

size_t mxfp4_scale_bytes(int64_t M, int64_t K) {
  if (M <= 0 || K <= 0 || K % 32 != 0 || M > kMaxRows) return 0;
  return rows_times_cols(ceil_div(M, 128) * 128, padded_scale_cols(K));
}

size_t mxfp4_grouped_scale_bytes_bound(int64_t total_rows, int32_t E, int64_t K) {
  if (total_rows < 0 || E < 0 || K <= 0 || K % 32 != 0 || total_rows > kMaxRows) return 0;
  const int64_t tiles = (total_rows + 127 * static_cast<int64_t>(E)) / 128;
  return rows_times_cols(tiles * 128, padded_scale_cols(K));
}

}  // extern "C"

namespace {

int quantize_checked(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes,
                     uint8_t* scales, bool f16, void* stream) {
  if (M < 0 || K < 0) return MXFP4_EINVAL;
  if (K % 32 != 0 || ldx < K) return MXFP4_ESHAPE;
  if (M == 0 || K == 0) return MXFP4_OK;
  if (!x || !codes || !scales) return MXFP4_EINVAL;
  if (!aligned16(x) || ldx % 8 != 0 || !aligned16(codes) || !aligned16(scales))
    return MXFP4_EALIGN;
  const int64_t tiles = ceil_div(M, 128) * ceil_div(K / 32, 4);
  if (M > (INT64_MAX / 4) / ldx || tiles > kMaxGrid) return MXFP4_ESHAPE;
  const Range rx = range_of(x, ((M - 1) * ldx + K) * 2);
  const Range rc = range_of(codes, M * (K / 2));
  const Range rs = range_of(scales, static_cast<int64_t>(mxfp4_scale_bytes(M, K)));
  if (overlap(rx, rc) || overlap(rx, rs) || overlap(rc, rs)) return MXFP4_EALIAS;
  return from_cuda(mxfp4::launch_quantize(x, M, K, ldx, codes, scales, f16,
                                          static_cast<cudaStream_t>(stream)));
}

int grouped_checked(const void* x, int64_t total_rows, int64_t K,
                           const int32_t* expert_offsets, int32_t E, uint8_t* codes,
                           uint8_t* scales, int32_t* scale_row_offsets, int32_t* status,
                    bool f16, void* stream) {
  if (total_rows < 0 || K < 0 || E < 0) return MXFP4_EINVAL;
  if (K % 32 != 0) return MXFP4_ESHAPE;
  if (!expert_offsets || !scale_row_offsets) return MXFP4_EINVAL;
  if (total_rows > 0 && K > 0 && (!x || !codes || !scales)) return MXFP4_EINVAL;
  if (E == 0 && total_rows > 0) return MXFP4_EINVAL;
  // padded rows must fit int32 (scale_row_offsets) and the grid must fit
  const int64_t bound_tiles = (total_rows + 127 * static_cast<int64_t>(E)) / 128;
  if (total_rows + 127 * static_cast<int64_t>(E) > INT32_MAX) return MXFP4_ESHAPE;
  const int64_t grid = bound_tiles * ceil_div(K / 32, 4);
  if (grid > kMaxGrid) return MXFP4_ESHAPE;
  if ((x && !aligned16(x)) || (codes && !aligned16(codes)) || (scales && !aligned16(scales)) ||
      (reinterpret_cast<uintptr_t>(expert_offsets) & 3u) ||
      (reinterpret_cast<uintptr_t>(scale_row_offsets) & 3u) ||
      (reinterpret_cast<uintptr_t>(status) & 3u))
    return MXFP4_EALIGN;
  const Range rx = range_of(x, total_rows * K * 2);
  const Range ro = range_of(expert_offsets, (static_cast<int64_t>(E) + 1) * 4);
  const Range rc = range_of(codes, total_rows * (K / 2));
  const Range rs =
      range_of(scales, static_cast<int64_t>(mxfp4_grouped_scale_bytes_bound(total_rows, E, K)));
  const Range rp = range_of(scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4);
  const Range rt = range_of(status, status ? 4 : 0);
  const Range outs[4] = {rc, rs, rp, rt};
  for (int i = 0; i < 4; ++i) {
    if (overlap(outs[i], rx) || overlap(outs[i], ro)) return MXFP4_EALIAS;
    for (int j = i + 1; j < 4; ++j)
      if (overlap(outs[i], outs[j])) return MXFP4_EALIAS;
  }
  const int64_t tiles = (K == 0) ? 0 : bound_tiles;
  return from_cuda(mxfp4::launch_quantize_grouped(x, total_rows, K, expert_offsets, E, codes,
                                                  scales, scale_row_offsets, status, tiles, f16,
                                                  static_cast<cudaStream_t>(stream)));
}

// How a gather call runs: the per-row gather kernel, or the scatter path with
// the inverse map in a workspace, its scale words stored straight into the
// tiled layout (kInverse) or staged per token and tiled by a second kernel
// (kInverseStaged, the larger workspace).  kScratch: the scatter path in the
// library's fixed scratch array, staged when the whole workspace fits it,
// else kInverse; MXFP4_ESCRATCH when not even the inverse map fits.
enum class GatherPath { kPerRow, kInverse, kInverseStaged, kScratch };

int64_t gather_ws_bytes(int64_t num_src_rows, int64_t total_rows, int32_t E, int64_t K,
                        bool staged) {
  const int64_t map = mxfp4::gather_workspace_ints(num_src_rows, total_rows) +
                      (staged ? mxfp4::gather_tok_ints(total_rows, E) : 0);
  return ceil_div(map * 4, 16) * 16 +
         (staged ? mxfp4::gather_stage_ints(num_src_rows, K) * 4 : 0);
}

int gather_checked(const void* x, int64_t num_src_rows, int64_t K, int64_t ldx,
                   const int32_t* row_index, int64_t total_rows, const int32_t* expert_offsets,
                   int32_t E, void* workspace, size_t workspace_bytes, uint8_t* codes,
                   uint8_t* scales, int32_t* scale_row_offsets, int32_t* status, GatherPath path,
                   bool f16, void* stream) {
  const bool use_ws = path != GatherPath::kPerRow;
  const bool in_scratch = path == GatherPath::kScratch;
  bool staged = path == GatherPath::kInverseStaged;
  if (num_src_rows < 0 || total_rows < 0 || K < 0 || E < 0) return MXFP4_EINVAL;
  if (K % 32 != 0 || ldx < K) return MXFP4_ESHAPE;
  if (!expert_offsets || !scale_row_offsets) return MXFP4_EINVAL;
  const bool work = total_rows > 0 && K > 0;
  if (work && (!x || !row_index || !codes || !scales || num_src_rows == 0)) return MXFP4_EINVAL;
  if (E == 0 && total_rows > 0) return MXFP4_EINVAL;
  const int64_t bound_tiles = (total_rows + 127 * static_cast<int64_t>(E)) / 128;
  if (total_rows + 127 * static_cast<int64_t>(E) > INT32_MAX) return MXFP4_ESHAPE;
  if (bound_tiles * ceil_div(K / 32, 4) > kMaxGrid) return MXFP4_ESHAPE;
  if (num_src_rows > 0 && ldx > 0 && num_src_rows > (INT64_MAX / 4) / ldx) return MXFP4_ESHAPE;
  int64_t ws_bytes = 0;
  if (use_ws) {
    // token ids and route counts are int32 on the device
    if (num_src_rows > INT32_MAX / 4) return MXFP4_ESHAPE;
    if (num_src_rows > (INT64_MAX / 8) / (K / 128 + 1)) return MXFP4_ESHAPE;
    if (in_scratch) {
      // the staged form when its whole workspace fits the library's array;
      // the array's address is looked up only for a call that fits it
      staged = gather_ws_bytes(num_src_rows, total_rows, E, K, true) <=
               static_cast<int64_t>(workspace_bytes);
      if (work && gather_ws_bytes(num_src_rows, total_rows, E, K, staged) >
                      static_cast<int64_t>(workspace_bytes))
        return MXFP4_ESCRATCH;
      if (work && (workspace = mxfp4::noalloc_scratch()) == nullptr) return MXFP4_ECUDA;
    }
    ws_bytes = gather_ws_bytes(num_src_rows, total_rows, E, K, staged);
    if (work && (!workspace || workspace_bytes < static_cast<size_t>(ws_bytes)))
      return MXFP4_EINVAL;
    if (workspace && !aligned16(workspace)) return MXFP4_EALIGN;
  }
  if ((x && (!aligned16(x) || ldx % 8 != 0)) || (codes && !aligned16(codes)) ||
      (scales && !aligned16(scales)) || (reinterpret_cast<uintptr_t>(row_index) & 3u) ||
      (reinterpret_cast<uintptr_t>(expert_offsets) & 3u) ||
      (reinterpret_cast<uintptr_t>(scale_row_offsets) & 3u) ||
      (reinterpret_cast<uintptr_t>(status) & 3u))
    return MXFP4_EALIGN;
  const Range ins[3] = {
      range_of(x, work ? ((num_src_rows - 1) * ldx + K) * 2 : 0),
      range_of(row_index, work ? total_rows * 4 : 0),
      range_of(expert_offsets, (static_cast<int64_t>(E) + 1) * 4)};
  const Range outs[5] = {
      range_of(codes, total_rows * (K / 2)),
      range_of(scales,
               static_cast<int64_t>(mxfp4_grouped_scale_bytes_bound(total_rows, E, K))),
      range_of(scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4),
      range_of(status, status ? 4 : 0),
      range_of(workspace, use_ws && work ? ws_bytes : 0)};
  for (int i = 0; i < 5; ++i) {
    for (int j = 0; j < 3; ++j)
      if (overlap(outs[i], ins[j])) return MXFP4_EALIAS;
    for (int j = i + 1; j < 5; ++j)
      if (overlap(outs[i], outs[j])) return MXFP4_EALIAS;
  }
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (use_ws)
    return from_cuda(mxfp4::launch_quantize_grouped_gather_ws(
        x, work ? num_src_rows : 0, K, ldx, row_index, total_rows, expert_offsets, E,
        static_cast<int32_t*>(workspace), staged, codes, scales, scale_row_offsets, status,
        K == 0 ? 0 : bound_tiles, f16, st));
  // no workspace: through the scatter path in the borrowed tail of the codes
  // output when it is large enough, else the per-row gather kernel
  if (work && E > 0 && num_src_rows <= INT32_MAX / 4 &&
      mxfp4::gather_borrow_rows(num_src_rows, total_rows, E, K) >= 0)
    return from_cuda(mxfp4::launch_quantize_grouped_gather_borrowed(
        x, num_src_rows, K, ldx, row_index, total_rows, expert_offsets, E, codes, scales,
        scale_row_offsets, status, bound_tiles, f16, st));
  return from_cuda(mxfp4::launch_quantize_grouped_gather(
      x, num_src_rows, K, ldx, row_index, total_rows, expert_offsets, E, codes, scales,
      scale_row_offsets, status, K == 0 ? 0 : bound_tiles, f16, st));
}

int scatter_checked(const void* x, int64_t num_tokens, int64_t K, int64_t ldx,
                    const int32_t* dest_rows, int32_t top_k, int64_t total_rows,
                    const int32_t* expert_offsets, int32_t E, void* workspace,
                    size_t workspace_bytes, bool use_ws, uint8_t* codes, uint8_t* scales,
                    int32_t* scale_row_offsets, int32_t* status, bool f16, void* stream) {
  if (num_tokens < 0 || total_rows < 0 || K < 0 || E < 0) return MXFP4_EINVAL;
  if (top_k < 1 || top_k > MXFP4_SCATTER_MAX_TOP_K) return MXFP4_EINVAL;
  if (K % 32 != 0 || ldx < K) return MXFP4_ESHAPE;
  if (!expert_offsets || !scale_row_offsets) return MXFP4_EINVAL;
  const bool rows = total_rows > 0 && K > 0;
  const bool reads = rows && num_tokens > 0;
  if (rows && (!codes || !scales)) return MXFP4_EINVAL;
  if (reads && (!x || !dest_rows)) return MXFP4_EINVAL;
  if (E == 0 && total_rows > 0) return MXFP4_EINVAL;
  const int64_t bound_tiles = (total_rows + 127 * static_cast<int64_t>(E)) / 128;
  if (total_rows + 127 * static_cast<int64_t>(E) > INT32_MAX) return MXFP4_ESHAPE;
  const int64_t n_chunks = ceil_div(ceil_div(K / 32, 4), 4);
  if (E + ceil_div(num_tokens, 128) * n_chunks > kMaxGrid) return MXFP4_ESHAPE;
  if (num_tokens > (INT64_MAX / 4) / (ldx > top_k ? ldx : top_k)) return MXFP4_ESHAPE;
  int64_t ws_bytes = 0;
  if (use_ws) {
    // token ids are int32 on the device
    if (num_tokens > INT32_MAX / 4) return MXFP4_ESHAPE;
    ws_bytes = mxfp4::scatter_workspace_ints(num_tokens, total_rows, E, K) * 4;
    if (rows && (!workspace || workspace_bytes < static_cast<size_t>(ws_bytes)))
      return MXFP4_EINVAL;
    if (workspace && !aligned16(workspace)) return MXFP4_EALIGN;
  }
  if ((x && (!aligned16(x) || ldx % 8 != 0)) || (codes && !aligned16(codes)) ||
      (scales && !aligned16(scales)) || (reinterpret_cast<uintptr_t>(dest_rows) & 3u) ||
      (reinterpret_cast<uintptr_t>(expert_offsets) & 3u) ||
      (reinterpret_cast<uintptr_t>(scale_row_offsets) & 3u) ||
      (reinterpret_cast<uintptr_t>(status) & 3u))
    return MXFP4_EALIGN;
  const Range ins[3] = {
      range_of(x, reads ? ((num_tokens - 1) * ldx + K) * 2 : 0),
      range_of(dest_rows, reads ? num_tokens * top_k * 4 : 0),
      range_of(expert_offsets, (static_cast<int64_t>(E) + 1) * 4)};
  const Range outs[5] = {
      range_of(codes, total_rows * (K / 2)),
      range_of(scales,
               static_cast<int64_t>(mxfp4_grouped_scale_bytes_bound(total_rows, E, K))),
      range_of(scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4),
      range_of(status, status ? 4 : 0),
      range_of(workspace, use_ws && rows ? ws_bytes : 0)};
  for (int i = 0; i < 5; ++i) {
    for (int j = 0; j < 3; ++j)
      if (overlap(outs[i], ins[j])) return MXFP4_EALIAS;
    for (int j = i + 1; j < 5; ++j)
      if (overlap(outs[i], outs[j])) return MXFP4_EALIAS;
  }
  return from_cuda(mxfp4::launch_quantize_grouped_scatter(
      x, reads ? num_tokens : 0, K, ldx, dest_rows, top_k, total_rows, expert_offsets, E,
      use_ws && rows ? static_cast<int32_t*>(workspace) : nullptr, codes, scales,
      scale_row_offsets, status, K == 0 ? 0 : bound_tiles, f16,
      static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

int mxfp4_quantize(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes,
                   uint8_t* scales, void* stream) {
  return quantize_checked(x, M, K, ldx, codes, scales, false, stream);
}

int mxfp4_quantize_f16(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes,
                       uint8_t* scales, void* stream) {
  return quantize_checked(x, M, K, ldx, codes, scales, true, stream);
}

int mxfp4_quantize_grouped(const void* x, int64_t total_rows, int64_t K,
                           const int32_t* expert_offsets, int32_t E, uint8_t* codes,
                           uint8_t* scales, int32_t* scale_row_offsets, int32_t* status,
                           void* stream) {
  return grouped_checked(x, total_rows, K, expert_offsets, E, codes, scales, scale_row_offsets,
                         status, false, stream);
}

int mxfp4_quantize_grouped_f16(const void* x, int64_t total_rows, int64_t K,
                               const int32_t* expert_offsets, int32_t E, uint8_t* codes,
                               uint8_t* scales, int32_t* scale_row_offsets, int32_t* status,
                               void* stream) {
  return grouped_checked(x, total_rows, K, expert_offsets, E, codes, scales, scale_row_offsets,
                         status, true, stream);
}

int mxfp4_quantize_grouped_gather(const void* x, int64_t num_src_rows, int64_t K, int64_t ldx,
                                  const int32_t* row_index, int64_t total_rows,
                                  const int32_t* expert_offsets, int32_t E, uint8_t* codes,
                                  uint8_t* scales, int32_t* scale_row_offsets, int32_t* status,
                                  void* stream) {
  return gather_checked(x, num_src_rows, K, ldx, row_index, total_rows, expert_offsets, E,
                        nullptr, 0, codes, scales, scale_row_offsets, status,
                        GatherPath::kPerRow, false, stream);
}

int mxfp4_quantize_grouped_gather_f16(const void* x, int64_t num_src_rows, int64_t K, int64_t ldx,
                                      const int32_t* row_index, int64_t total_rows,
                                      const int32_t* expert_offsets, int32_t E, uint8_t* codes,
                                      uint8_t* scales, int32_t* scale_row_offsets,
                                      int32_t* status, void* stream) {
  return gather_checked(x, num_src_rows, K, ldx, row_index, total_rows, expert_offsets, E,
                        nullptr, 0, codes, scales, scale_row_offsets, status,
                        GatherPath::kPerRow, true, stream);
}

size_t mxfp4_gather_workspace_bytes(int64_t num_src_rows, int64_t total_rows, int32_t E,
                                    int64_t K) {
  if (num_src_rows < 0 || total_rows < 0 || E < 0 || K < 0 || K % 32 != 0) return 0;
  if (num_src_rows > INT32_MAX / 4 || total_rows + 127 * static_cast<int64_t>(E) > INT32_MAX)
    return 0;
  // the same bounds the calls apply: k tiles and staged words stay countable
  if (ceil_div(K / 32, 4) > kMaxGrid || num_src_rows > (INT64_MAX / 8) / (K / 128 + 1)) return 0;
  return static_cast<size_t>(gather_ws_bytes(num_src_rows, total_rows, E, K, K > 0));
}

int mxfp4_quantize_grouped_gather_ws(const void* x, int64_t num_src_rows, int64_t K, int64_t ldx,
                                     const int32_t* row_index, int64_t total_rows,
                                     const int32_t* expert_offsets, int32_t E, void* workspace,
                                     size_t workspace_bytes, uint8_t* codes, uint8_t* scales,
                                     int32_t* scale_row_offsets, int32_t* status, void* stream) {
  return gather_checked(x, num_src_rows, K, ldx, row_index, total_rows, expert_offsets, E,
                        workspace, workspace_bytes, codes, scales, scale_row_offsets, status,
                        GatherPath::kInverseStaged, false, stream);
}

int mxfp4_quantize_grouped_gather_noalloc(const void* x, int64_t num_src_rows, int64_t K,
                                          int64_t ldx, const int32_t* row_index,
                                          int64_t total_rows, const int32_t* expert_offsets,
                                          int32_t E, uint8_t* codes, uint8_t* scales,
                                          int32_t* scale_row_offsets, int32_t* status,
                                          void* stream) {
  return gather_checked(x, num_src_rows, K, ldx, row_index, total_rows, expert_offsets, E,
                        nullptr, MXFP4_NOALLOC_SCRATCH_BYTES, codes, scales, scale_row_offsets,
                        status, GatherPath::kScratch, false, stream);
}

int mxfp4_quantize_grouped_gather_ws_f16(const void* x, int64_t num_src_rows, int64_t K,
                                         int64_t ldx, const int32_t* row_index,
                                         int64_t total_rows, const int32_t* expert_offsets,
                                         int32_t E, void* workspace, size_t workspace_bytes,
                                         uint8_t* codes, uint8_t* scales,
                                         int32_t* scale_row_offsets, int32_t* status,
                                         void* stream) {
  return gather_checked(x, num_src_rows, K, ldx, row_index, total_rows, expert_offsets, E,
                        workspace, workspace_bytes, codes, scales, scale_row_offsets, status,
                        GatherPath::kInverseStaged, true, stream);
}

int mxfp4_quantize_grouped_scatter(const void* x, int64_t num_tokens, int64_t K, int64_t ldx,
                                   const int32_t* dest_rows, int32_t top_k, int64_t total_rows,
                                   const int32_t* expert_offsets, int32_t E, uint8_t* codes,
                                   uint8_t* scales, int32_t* scale_row_offsets, int32_t* status,
                                   void* stream) {
  return scatter_checked(x, num_tokens, K, ldx, dest_rows, top_k, total_rows, expert_offsets, E,
                         nullptr, 0, false, codes, scales, scale_row_offsets, status, false,
                         stream);
}

int mxfp4_quantize_grouped_scatter_f16(const void* x, int64_t num_tokens, int64_t K, int64_t ldx,
                                       const int32_t* dest_rows, int32_t top_k,
                                       int64_t total_rows, const int32_t* expert_offsets,
                                       int32_t E, uint8_t* codes, uint8_t* scales,
                                       int32_t* scale_row_offsets, int32_t* status,
                                       void* stream) {
  return scatter_checked(x, num_tokens, K, ldx, dest_rows, top_k, total_rows, expert_offsets, E,
                         nullptr, 0, false, codes, scales, scale_row_offsets, status, true,
                         stream);
}

size_t mxfp4_scatter_workspace_bytes(int64_t num_tokens, int64_t total_rows, int32_t E,
                                     int64_t K) {
  if (num_tokens < 0 || total_rows < 0 || E < 0 || K < 0 || K % 32 != 0) return 0;
  if (num_tokens > INT32_MAX / 4 || total_rows + 127 * static_cast<int64_t>(E) > INT32_MAX)
    return 0;
  // the k-tile bound the calls apply (the staged rows count k tiles in int)
  if (ceil_div(K / 32, 4) > kMaxGrid) return 0;
  return static_cast<size_t>(mxfp4::scatter_workspace_ints(num_tokens, total_rows, E, K) * 4);
}

int mxfp4_quantize_grouped_scatter_ws(const void* x, int64_t num_tokens, int64_t K, int64_t ldx,
                                      const int32_t* dest_rows, int32_t top_k,
                                      int64_t total_rows, const int32_t* expert_offsets,
                                      int32_t E, void* workspace, size_t workspace_bytes,
                                      uint8_t* codes, uint8_t* scales,
                                      int32_t* scale_row_offsets, int32_t* status,
                                      void* stream) {
  return scatter_checked(x, num_tokens, K, ldx, dest_rows, top_k, total_rows, expert_offsets, E,
                         workspace, workspace_bytes, true, codes, scales, scale_row_offsets,
                         status, false, stream);
}

int mxfp4_quantize_grouped_scatter_ws_f16(const void* x, int64_t num_tokens, int64_t K,
                                          int64_t ldx, const int32_t* dest_rows, int32_t top_k,
                                          int64_t total_rows, const int32_t* expert_offsets,
                                          int32_t E, void* workspace, size_t workspace_bytes,
                                          uint8_t* codes, uint8_t* scales,
                                          int32_t* scale_row_offsets, int32_t* status,
                                          void* stream) {
  return scatter_checked(x, num_tokens, K, ldx, dest_rows, top_k, total_rows, expert_offsets, E,
                         workspace, workspace_bytes, true, codes, scales, scale_row_offsets,
                         status, true, stream);
}




int mxfp4_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t M, int64_t K, void* y,
                     void* stream) {
  if (M < 0 || K < 0) return MXFP4_EINVAL;
  if (K % 32 != 0) return MXFP4_ESHAPE;
  if (M == 0 || K == 0) return MXFP4_OK;
  if (!codes || !scales || !y) return MXFP4_EINVAL;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(y)) return MXFP4_EALIGN;
  const int64_t tiles = ceil_div(M, 128) * ceil_div(K / 32, 4);
  if (M > (INT64_MAX / 4) / K || tiles > kMaxGrid) return MXFP4_ESHAPE;
  const Range rc = range_of(codes, M * (K / 2));
  const Range rs = range_of(scales, static_cast<int64_t>(mxfp4_scale_bytes(M, K)));
  const Range ry = range_of(y, M * K * 2);
  if (overlap(ry, rc) || overlap(ry, rs)) return MXFP4_EALIAS;
  return from_cuda(
      mxfp4::launch_dequantize(codes, scales, M, K, y, static_cast<cudaStream_t>(stream)));
}

size_t mxfp4_route_workspace_bytes(int64_t num_tokens, int32_t top_k, int32_t E) {
  if (num_tokens < 0 || top_k < 1 || E < 1 || E > MXFP4_ROUTE_MAX_EXPERTS) return 0;
  if (num_tokens > (INT32_MAX / 2) / top_k) return 0;
  return static_cast<size_t>(mxfp4::route_workspace_ints(num_tokens * top_k, E) * 4);
}

int mxfp4_moe_route(const int32_t* topk_ids, int64_t num_tokens, int32_t top_k, int32_t E,
                    void* workspace, size_t workspace_bytes, int32_t* expert_offsets,
                    int32_t* dest_rows, int32_t* row_index, int32_t* status, void* stream) {
  if (num_tokens < 0 || top_k < 1 || E < 1) return MXFP4_EINVAL;
  if (E > MXFP4_ROUTE_MAX_EXPERTS || num_tokens > (INT32_MAX / 2) / top_k) return MXFP4_ESHAPE;
  const int64_t n = num_tokens * top_k;
  if (!expert_offsets || (n > 0 && (!topk_ids || !dest_rows))) return MXFP4_EINVAL;
  const int64_t ws_bytes = mxfp4::route_workspace_ints(n, E) * 4;
  if (n > 0 && (!workspace || workspace_bytes < static_cast<size_t>(ws_bytes)))
    return MXFP4_EINVAL;
  const auto misaligned4 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 3u) != 0; };
  if (misaligned4(topk_ids) || misaligned4(expert_offsets) || misaligned4(dest_rows) ||
      misaligned4(row_index) || misaligned4(status) || (workspace && !aligned16(workspace)))
    return MXFP4_EALIGN;
  const Range in = range_of(topk_ids, n * 4);
  const Range outs[5] = {range_of(expert_offsets, (static_cast<int64_t>(E) + 1) * 4),
                         range_of(dest_rows, n * 4), range_of(row_index, row_index ? n * 4 : 0),
                         range_of(status, status ? 4 : 0),
                         range_of(workspace, n > 0 ? ws_bytes : 0)};
  for (int i = 0; i < 5; ++i) {
    if (overlap(outs[i], in)) return MXFP4_EALIAS;
    for (int j = i + 1; j < 5; ++j)
      if (overlap(outs[i], outs[j])) return MXFP4_EALIAS;
  }
  return from_cuda(mxfp4::launch_moe_route(topk_ids, num_tokens, top_k, E,
                                           static_cast<int32_t*>(workspace), expert_offsets,
                                           dest_rows, row_index, status,
                                           static_cast<cudaStream_t>(stream)));
}

int mxfp4_swap_w13(const uint8_t* codes_in, const uint8_t* scales_in, const float* w13_bias_in,
                   int32_t E, int64_t two_n, int64_t K, int32_t scales_tiled, uint8_t* codes_out,
                   uint8_t* scales_out, void* w13_bias_out, const float* w2_bias_in,
                   int64_t w2_bias_numel, void* w2_bias_out, void* stream) {
  if (E < 0 || two_n < 0 || K < 0 || w2_bias_numel < 0) return MXFP4_EINVAL;
  if (scales_tiled != 0 && scales_tiled != 1) return MXFP4_EINVAL;
  if (two_n % 2 != 0 || K % 32 != 0) return MXFP4_ESHAPE;
  const bool w13_work = E > 0 && two_n > 0 && K > 0;
  if (w13_work && (!codes_in || !scales_in || !codes_out || !scales_out)) return MXFP4_EINVAL;
  if (w13_bias_in && E > 0 && two_n > 0 && !w13_bias_out) return MXFP4_EINVAL;
  if (w2_bias_in && w2_bias_numel > 0 && !w2_bias_out) return MXFP4_EINVAL;
  if (static_cast<int64_t>(E) * two_n > INT64_MAX / (K > 0 ? K : 1) / 4) return MXFP4_ESHAPE;
  if ((codes_in && !aligned16(codes_in)) || (codes_out && !aligned16(codes_out)) ||
      (scales_in && !aligned16(scales_in)) || (scales_out && !aligned16(scales_out)) ||
      (w13_bias_in && (reinterpret_cast<uintptr_t>(w13_bias_in) & 3u)) ||
      (w13_bias_out && (reinterpret_cast<uintptr_t>(w13_bias_out) & 1u)) ||
      (w2_bias_in && (reinterpret_cast<uintptr_t>(w2_bias_in) & 3u)) ||
      (w2_bias_out && (reinterpret_cast<uintptr_t>(w2_bias_out) & 1u)))
    return MXFP4_EALIGN;
  const int64_t rows = static_cast<int64_t>(E) * two_n;
  const int64_t scale_bytes =
      scales_tiled ? static_cast<int64_t>(E) * static_cast<int64_t>(mxfp4_scale_bytes(two_n, K))
                   : rows * (K / 32);
  const int64_t n13 = w13_bias_in ? rows : 0;
  const int64_t n2 = w2_bias_in ? w2_bias_numel : 0;
  const Range ins[4] = {range_of(codes_in, w13_work ? rows * (K / 2) : 0),
                        range_of(scales_in, w13_work ? scale_bytes : 0),
                        range_of(w13_bias_in, n13 * 4), range_of(w2_bias_in, n2 * 4)};
  const Range outs[4] = {range_of(codes_out, w13_work ? rows * (K / 2) : 0),
                         range_of(scales_out, w13_work ? scale_bytes : 0),
                         range_of(w13_bias_out, n13 * 2), range_of(w2_bias_out, n2 * 2)};
  for (int i = 0; i < 4; ++i) {
    for (int j = 0; j < 4; ++j)
      if (overlap(outs[i], ins[j])) return MXFP4_EALIAS;
    for (int j = i + 1; j < 4; ++j)
      if (overlap(outs[i], outs[j])) return MXFP4_EALIAS;
  }
  mxfp4::SwapArgs a{};
  a.codes_in = codes_in;
  a.scales_in = scales_in;
  a.w13_bias_in = (E > 0 && two_n > 0) ? w13_bias_in : nullptr;
  a.E = w13_work ? E : 0;
  a.two_n = two_n > 0 ? two_n : 2;
  a.K = K;
  a.scales_tiled = scales_tiled;
  a.codes_out = codes_out;
  a.scales_out = scales_out;
  a.w13_bias_out = w13_bias_out;
  a.w2_bias_in = n2 > 0 ? w2_bias_in : nullptr;
  a.w2_bias_numel = n2;
  a.w2_bias_out = w2_bias_out;
  if (!w13_work) {
    // bias-only work (e.g. K == 0): keep the bias part, skip codes/scales
    a.E = (E > 0 && two_n > 0) ? E : 0;
    a.K = 0;
  }
  if (a.E == 0 && n2 == 0) return MXFP4_OK;
  return from_cuda(mxfp4::launch_swap_w13(a, static_cast<cudaStream_t>(stream)));
}

size_t mxfp4_nvfp4_scale_bytes(int64_t M, int64_t K) {
  if (M <= 0 || K <= 0 || K % 16 != 0 || M > kMaxRows) return 0;
  return rows_times_cols(ceil_div(M, 128) * 128, ceil_div(K / 16, 4) * 4);
}

}  // extern "C"

namespace {

int nvfp4_checked(const void* x, int64_t M, int64_t K, int64_t ldx, const float* global_scale,
                  uint8_t* codes, uint8_t* scales, bool f16, void* stream) {
  if (M < 0 || K < 0) return MXFP4_EINVAL;
  if (K % 16 != 0 || ldx < K) return MXFP4_ESHAPE;
  if (M == 0 || K == 0) return MXFP4_OK;
  if (!x || !global_scale || !codes || !scales) return MXFP4_EINVAL;
  if (!aligned16(x) || ldx % 8 != 0 || !aligned16(codes) || !aligned16(scales) ||
      (reinterpret_cast<uintptr_t>(global_scale) & 3u))
    return MXFP4_EALIGN;
  const int64_t ctas = ceil_div(M, 128) * ceil_div(ceil_div(K / 16, 4), 2);
  if (M > (INT64_MAX / 4) / ldx || ctas > kMaxGrid) return MXFP4_ESHAPE;
  const Range rx = range_of(x, ((M - 1) * ldx + K) * 2);
  const Range rg = range_of(global_scale, 4);
  const Range rc = range_of(codes, M * (K / 2));
  const Range rs = range_of(scales, static_cast<int64_t>(mxfp4_nvfp4_scale_bytes(M, K)));
  if (overlap(rx, rc) || overlap(rx, rs) || overlap(rc, rs) || overlap(rg, rc) ||
      overlap(rg, rs))
    return MXFP4_EALIAS;
  return from_cuda(mxfp4::launch_quantize_nvfp4(x, M, K, ldx, global_scale, codes, scales, f16,
                                                static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

int mxfp4_quantize_nvfp4(const void* x, int64_t M, int64_t K, int64_t ldx,
                         const float* global_scale, uint8_t* codes, uint8_t* scales,
                         void* stream) {
  return nvfp4_checked(x, M, K, ldx, global_scale, codes, scales, false, stream);
}

int mxfp4_quantize_nvfp4_f16(const void* x, int64_t M, int64_t K, int64_t ldx,
                             const float* global_scale, uint8_t* codes, uint8_t* scales,
                             void* stream) {
  return nvfp4_checked(x, M, K, ldx, global_scale, codes, scales, true, stream);
}

size_t mxfp4_nvfp4_grouped_scale_bytes_bound(int64_t total_rows, int32_t E, int64_t K) {
  if (total_rows < 0 || E < 0 || K <= 0 || K % 16 != 0 || total_rows > kMaxRows) return 0;
  const int64_t tiles = (total_rows + 127 * static_cast<int64_t>(E)) / 128;
  return rows_times_cols(tiles * 128, ceil_div(K / 16, 4) * 4);
}

}  // extern "C"

namespace {

int nvfp4_grouped_checked(const void* x, int64_t total_rows, int64_t K,
                          const int32_t* expert_offsets, int32_t E, const float* global_scales,
                          uint8_t* codes, uint8_t* scales, int32_t* scale_row_offsets,
                          int32_t* status, bool f16, void* stream) {
  if (total_rows < 0 || K < 0 || E < 0) return MXFP4_EINVAL;
  if (K % 16 != 0) return MXFP4_ESHAPE;
  if (!expert_offsets || !scale_row_offsets) return MXFP4_EINVAL;
  const bool work = total_rows > 0 && K > 0;
  if (work && (!x || !codes || !scales || !global_scales)) return MXFP4_EINVAL;
  if (E == 0 && total_rows > 0) return MXFP4_EINVAL;
  const int64_t bound_tiles = (total_rows + 127 * static_cast<int64_t>(E)) / 128;
  if (total_rows + 127 * static_cast<int64_t>(E) > INT32_MAX) return MXFP4_ESHAPE;
  if (bound_tiles * ceil_div(ceil_div(K / 16, 4), 2) > kMaxGrid) return MXFP4_ESHAPE;
  if (total_rows > 0 && K > 0 && total_rows > (INT64_MAX / 4) / K) return MXFP4_ESHAPE;
  if ((x && !aligned16(x)) || (codes && !aligned16(codes)) || (scales && !aligned16(scales)) ||
      (reinterpret_cast<uintptr_t>(global_scales) & 3u) ||
      (reinterpret_cast<uintptr_t>(expert_offsets) & 3u) ||
      (reinterpret_cast<uintptr_t>(scale_row_offsets) & 3u) ||
      (reinterpret_cast<uintptr_t>(status) & 3u))
    return MXFP4_EALIGN;
  const Range ins[3] = {range_of(x, work ? total_rows * K * 2 : 0),
                        range_of(global_scales, work ? static_cast<int64_t>(E) * 4 : 0),
                        range_of(expert_offsets, (static_cast<int64_t>(E) + 1) * 4)};
  const Range outs[4] = {
      range_of(codes, total_rows * (K / 2)),
      range_of(scales,
               static_cast<int64_t>(mxfp4_nvfp4_grouped_scale_bytes_bound(total_rows, E, K))),
      range_of(scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4),
      range_of(status, status ? 4 : 0)};
  for (int i = 0; i < 4; ++i) {
    for (int j = 0; j < 3; ++j)
      if (overlap(outs[i], ins[j])) return MXFP4_EALIAS;
    for (int j = i + 1; j < 4; ++j)
      if (overlap(outs[i], outs[j])) return MXFP4_EALIAS;
  }
  return from_cuda(mxfp4::launch_quantize_nvfp4_grouped(
      x, total_rows, K, expert_offsets, E, global_scales, codes, scales, scale_row_offsets,
      status, K == 0 ? 0 : bound_tiles, f16, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

int mxfp4_quantize_nvfp4_grouped(const void* x, int64_t total_rows, int64_t K,
                                 const int32_t* expert_offsets, int32_t E,
                                 const float* global_scales, uint8_t* codes, uint8_t* scales,
                                 int32_t* scale_row_offsets, int32_t* status, void* stream) {
  return nvfp4_grouped_checked(x, total_rows, K, expert_offsets, E, global_scales, codes, scales,
                               scale_row_offsets, status, false, stream);
}

int mxfp4_quantize_nvfp4_grouped_f16(const void* x, int64_t total_rows, int64_t K,
                                     const int32_t* expert_offsets, int32_t E,
                                     const float* global_scales, uint8_t* codes,
                                     uint8_t* scales, int32_t* scale_row_offsets,
                                     int32_t* status, void* stream) {
  return nvfp4_grouped_checked(x, total_rows, K, expert_offsets, E, global_scales, codes, scales,
                               scale_row_offsets, status, true, stream);
}

}  // extern "C"

namespace {

int nvfp4_scatter_checked(const void* x, int64_t num_tokens, int64_t K, int64_t ldx,
                          const int32_t* dest_rows, int32_t top_k, int64_t total_rows,
                          const int32_t* expert_offsets, int32_t E, const float* global_scales,
                          void* workspace, size_t workspace_bytes, bool use_ws, uint8_t* codes,
                          uint8_t* scales, int32_t* scale_row_offsets, int32_t* status, bool f16,
                          void* stream) {
  if (num_tokens < 0 || total_rows < 0 || K < 0 || E < 0) return MXFP4_EINVAL;
  if (top_k < 1 || top_k > MXFP4_SCATTER_MAX_TOP_K) return MXFP4_EINVAL;
  if (K % 16 != 0 || ldx < K) return MXFP4_ESHAPE;
  if (!expert_offsets || !scale_row_offsets) return MXFP4_EINVAL;
  const bool rows = total_rows > 0 && K > 0;
  const bool reads = rows && num_tokens > 0;
  if (rows && (!codes || !scales || !global_scales)) return MXFP4_EINVAL;
  if (reads && (!x || !dest_rows)) return MXFP4_EINVAL;
  if (E == 0 && total_rows > 0) return MXFP4_EINVAL;
  const int64_t bound_tiles = (total_rows + 127 * static_cast<int64_t>(E)) / 128;
  if (total_rows + 127 * static_cast<int64_t>(E) > INT32_MAX) return MXFP4_ESHAPE;
  if (E + ceil_div(num_tokens, 8) > kMaxGrid) return MXFP4_ESHAPE;
  if (num_tokens > (INT64_MAX / 4) / (ldx > top_k ? ldx : top_k)) return MXFP4_ESHAPE;
  int64_t ws_bytes = 0;
  if (use_ws) {
    ws_bytes = mxfp4::nvfp4_scatter_workspace_ints(total_rows, E, K) * 4;
    if (rows && (!workspace || workspace_bytes < static_cast<size_t>(ws_bytes)))
      return MXFP4_EINVAL;
    if (workspace && !aligned16(workspace)) return MXFP4_EALIGN;
  }
  if ((x && (!aligned16(x) || ldx % 8 != 0)) || (codes && !aligned16(codes)) ||
      (scales && !aligned16(scales)) || (reinterpret_cast<uintptr_t>(dest_rows) & 3u) ||
      (reinterpret_cast<uintptr_t>(global_scales) & 3u) ||
      (reinterpret_cast<uintptr_t>(expert_offsets) & 3u) ||
      (reinterpret_cast<uintptr_t>(scale_row_offsets) & 3u) ||
      (reinterpret_cast<uintptr_t>(status) & 3u))
    return MXFP4_EALIGN;
  const Range ins[4] = {
      range_of(x, reads ? ((num_tokens - 1) * ldx + K) * 2 : 0),
      range_of(dest_rows, reads ? num_tokens * top_k * 4 : 0),
      range_of(expert_offsets, (static_cast<int64_t>(E) + 1) * 4),
      range_of(global_scales, rows ? static_cast<int64_t>(E) * 4 : 0)};
  const Range outs[5] = {
      range_of(codes, total_rows * (K / 2)),
      range_of(scales,
               static_cast<int64_t>(mxfp4_nvfp4_grouped_scale_bytes_bound(total_rows, E, K))),
      range_of(scale_row_offsets, (static_cast<int64_t>(E) + 1) * 4),
      range_of(status, status ? 4 : 0),
      range_of(workspace, use_ws && rows ? ws_bytes : 0)};
  for (int i = 0; i < 5; ++i) {
    for (int j = 0; j < 4; ++j)
      if (overlap(outs[i], ins[j])) return MXFP4_EALIAS;
    for (int j = i + 1; j < 5; ++j)
      if (overlap(outs[i], outs[j])) return MXFP4_EALIAS;
  }
  return from_cuda(mxfp4::launch_quantize_nvfp4_grouped_scatter(
      x, reads ? num_tokens : 0, K, ldx, dest_rows, top_k, total_rows, expert_offsets, E,
      global_scales, use_ws && rows ? static_cast<int32_t*>(workspace) : nullptr, codes, scales,
      scale_row_offsets, status, K == 0 ? 0 : bound_tiles, f16,
      static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

int mxfp4_quantize_nvfp4_grouped_scatter(const void* x, int64_t num_tokens, int64_t K,
                                         int64_t ldx, const int32_t* dest_rows, int32_t top_k,
                                         int64_t total_rows, const int32_t* expert_offsets,
                                         int32_t E, const float* global_scales, uint8_t* codes,
                                         uint8_t* scales, int32_t* scale_row_offsets,
                                         int32_t* status, void* stream) {
  return nvfp4_scatter_checked(x, num_tokens, K, ldx, dest_rows, top_k, total_rows,
                               expert_offsets, E, global_scales, nullptr, 0, false, codes, scales,
                               scale_row_offsets, status, false, stream);
}

int mxfp4_quantize_nvfp4_grouped_scatter_f16(const void* x, int64_t num_tokens, int64_t K,
                                             int64_t ldx, const int32_t* dest_rows,
                                             int32_t top_k, int64_t total_rows,
                                             const int32_t* expert_offsets, int32_t E,
                                             const float* global_scales, uint8_t* codes,
                                             uint8_t* scales, int32_t* scale_row_offsets,
                                             int32_t* status, void* stream) {
  return nvfp4_scatter_checked(x, num_tokens, K, ldx, dest_rows, top_k, total_rows,
                               expert_offsets, E, global_scales, nullptr, 0, false, codes, scales,
                               scale_row_offsets, status, true, stream);
}

size_t mxfp4_nvfp4_scatter_workspace_bytes(int64_t total_rows, int32_t E, int64_t K) {
  if (total_rows < 0 || E < 0 || K < 0 || K % 16 != 0) return 0;
  if (total_rows + 127 * static_cast<int64_t>(E) > INT32_MAX) return 0;
  if (ceil_div(K / 16, 4) > kMaxGrid) return 0;  // as the calls: k tiles counted in int
  return static_cast<size_t>(mxfp4::nvfp4_scatter_workspace_ints(total_rows, E, K) * 4);
}

int mxfp4_quantize_nvfp4_grouped_scatter_ws(const void* x, int64_t num_tokens, int64_t K,
                                            int64_t ldx, const int32_t* dest_rows, int32_t top_k,
                                            int64_t total_rows, const int32_t* expert_offsets,
                                            int32_t E, const float* global_scales,
                                            void* workspace, size_t workspace_bytes,
                                            uint8_t* codes, uint8_t* scales,
                                            int32_t* scale_row_offsets, int32_t* status,
                                            void* stream) {
  return nvfp4_scatter_checked(x, num_tokens, K, ldx, dest_rows, top_k, total_rows,
                               expert_offsets, E, global_scales, workspace, workspace_bytes, true,
                               codes, scales, scale_row_offsets, status, false, stream);
}

int mxfp4_quantize_nvfp4_grouped_scatter_ws_f16(const void* x, int64_t num_tokens, int64_t K,
                                                int64_t ldx, const int32_t* dest_rows,
                                                int32_t top_k, int64_t total_rows,
                                                const int32_t* expert_offsets, int32_t E,
                                                const float* global_scales, void* workspace,
                                                size_t workspace_bytes, uint8_t* codes,
                                                uint8_t* scales, int32_t* scale_row_offsets,
                                                int32_t* status, void* stream) {
  return nvfp4_scatter_checked(x, num_tokens, K, ldx, dest_rows, top_k, total_rows,
                               expert_offsets, E, global_scales, workspace, workspace_bytes, true,
                               codes, scales, scale_row_offsets, status, true, stream);
}

int mxfp4_dequantize_nvfp4(const uint8_t* codes, const uint8_t* scales, const float* global_scale,
                           int64_t M, int64_t K, void* y, void* stream) {
  if (M < 0 || K < 0) return MXFP4_EINVAL;
  if (K % 16 != 0) return MXFP4_ESHAPE;
  if (M == 0 || K == 0) return MXFP4_OK;
  if (!codes || !scales || !global_scale || !y) return MXFP4_EINVAL;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(y) ||
      (reinterpret_cast<uintptr_t>(global_scale) & 3u))
    return MXFP4_EALIGN;
  const int64_t ctas = ceil_div(M, 128) * ceil_div(ceil_div(K / 16, 4), 2);
  if (M > (INT64_MAX / 4) / K || ctas > kMaxGrid) return MXFP4_ESHAPE;
  const Range ry = range_of(y, M * K * 2);
  if (overlap(ry, range_of(codes, M * (K / 2))) ||
      overlap(ry, range_of(scales, static_cast<int64_t>(mxfp4_nvfp4_scale_bytes(M, K)))) ||
      overlap(ry, range_of(global_scale, 4)))
    return MXFP4_EALIAS;
  return from_cuda(mxfp4::launch_dequantize_nvfp4(codes, scales, global_scale, M, K, y,
                                                  static_cast<cudaStream_t>(stream)));
}

const char* mxfp4_status_string(int status) {
  switch (status) {
    case MXFP4_OK: return "MXFP4_OK: success";
    case MXFP4_EINVAL: return "MXFP4_EINVAL: NULL pointer, negative size or bad flag";
    case MXFP4_EALIGN: return "MXFP4_EALIGN: pointer or row stride breaks the 16-byte rule";
    case MXFP4_ESHAPE: return "MXFP4_ESHAPE: K % 32 != 0, ldx < K, odd two_n or size overflow";
    case MXFP4_EALIAS: return "MXFP4_EALIAS: an output overlaps an input or another output";
    case MXFP4_ECUDA: return "MXFP4_ECUDA: kernel launch failed";
    case MXFP4_EOFFSETS: return "MXFP4_EOFFSETS: expert offsets are not 0 <= ... <= total_rows";
    case MXFP4_EINDEX:
      return "MXFP4_EINDEX: a gather row index is outside [0, num_src_rows) or a scatter entry "
             "outside [-1, total_rows)";
    case MXFP4_ESCRATCH:
      return "MXFP4_ESCRATCH: the call needs more than the library's fixed scratch buffer "
             "(MXFP4_NOALLOC_SCRATCH_BYTES); use mxfp4_quantize_grouped_gather_ws";
    default: return "unknown mxfp4 status";
  }
}

int mxfp4_version(void) { return 100; }

#ifdef MXFP4_DEBUG_BOUNDS
int64_t mxfp4_debug_bounds_violations(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  return static_cast<int64_t>(mxfp4::debug_violations_quantize()) +
         mxfp4::debug_violations_dispatch() +
         mxfp4::debug_violations_dequantize() + mxfp4::debug_violations_nvfp4() +
         mxfp4::debug_violations_swap() + mxfp4::debug_violations_route();
}
#endif

}  // extern "C"
