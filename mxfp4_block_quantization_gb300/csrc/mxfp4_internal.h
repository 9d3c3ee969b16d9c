// mxfp4_internal.h — launchers shared between the kernel translation units
// and the C ABI (mxfp4_api.cu).  Arguments are already validated by the
// caller; each launcher only enqueues work and returns the launch status.
#pragma once

#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

namespace mxfp4 {

// Dense quantize of a [M, K] BF16 (or, with f16, IEEE binary16) matrix
// (row stride ldx elements).
cudaError_t launch_quantize(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* codes,
                            uint8_t* scales, bool f16, cudaStream_t stream);

// Grouped quantize: validates offsets and writes padded row starts, then
// quantizes every segment.  `bound_tiles` is the host-side upper bound of
// padded 128-row tiles.  With f16 the input is IEEE binary16 instead of
// BF16 (here and in the gather and scatter forms).
cudaError_t launch_quantize_grouped(const void* x, int64_t total_rows, int64_t K,
                                    const int32_t* offsets, int32_t E, uint8_t* codes,
                                    uint8_t* scales, int32_t* scale_row_offsets,
                                    int32_t* status, int64_t bound_tiles, bool f16,
                                    cudaStream_t stream);

// Validates expert offsets and writes the padded row starts P[0..E] (and
// the status word) on the device; every grouped launcher runs it first.
cudaError_t launch_offsets(const int32_t* offsets, int32_t E, int64_t total_rows,
                           int32_t* scale_row_offsets, int32_t* status, cudaStream_t stream);

// Grouped quantize of gathered rows: output row r reads source row
// row_index[r] of x (row stride ldx elements, num_src_rows rows).
cudaError_t launch_quantize_grouped_gather(const void* x, int64_t num_src_rows, int64_t K,
                                           int64_t ldx, const int32_t* row_index,
                                           int64_t total_rows, const int32_t* offsets, int32_t E,
                                           uint8_t* codes, uint8_t* scales,
                                           int32_t* scale_row_offsets, int32_t* status,
                                           int64_t bound_tiles, bool f16, cudaStream_t stream);
// The same gather through the scatter path: the inverse map is built in
// `workspace` (gather_workspace_ints(num_src_rows, total_rows) int32).  With
// `staged`, the workspace also holds gather_tok_ints(total_rows, E) int32
// (the token of every padded row) and, from the next 16-byte boundary,
// gather_stage_ints(num_src_rows, K) int32: the scatter then stores each
// token's scale words there once and a tile kernel writes the tiled scales
// whole; without it the scatter stores every row's scale words into the tiled
// layout itself.
int64_t gather_workspace_ints(int64_t num_src_rows, int64_t total_rows);
// The gather without a workspace can borrow the last gather_borrow_rows(...)
// rows of its codes output (at most a quarter of them; -1 when they do not
// suffice): those rows hold the staged workspace until their own codes are
// written last.  Same results as the other gather forms.
int64_t gather_borrow_rows(int64_t num_src_rows, int64_t total_rows, int64_t E, int64_t K);
cudaError_t launch_quantize_grouped_gather_borrowed(const void* x, int64_t num_src_rows,
                                                    int64_t K, int64_t ldx,
                                                    const int32_t* row_index, int64_t total_rows,
                                                    const int32_t* offsets, int32_t E,
                                                    uint8_t* codes, uint8_t* scales,
                                                    int32_t* scale_row_offsets, int32_t* status,
                                                    int64_t bound_tiles, bool f16,
                                                    cudaStream_t stream);
int64_t gather_tok_ints(int64_t total_rows, int64_t E);
int64_t gather_stage_ints(int64_t num_src_rows, int64_t K);
cudaError_t launch_quantize_grouped_gather_ws(const void* x, int64_t num_src_rows, int64_t K,
                                              int64_t ldx, const int32_t* row_index,
                                              int64_t total_rows, const int32_t* offsets,
                                              int32_t E, int32_t* workspace, bool staged,
                                              uint8_t* codes, uint8_t* scales,
                                              int32_t* scale_row_offsets, int32_t* status,
                                              int64_t bound_tiles, bool f16, cudaStream_t stream);
// The scatter (token -> rows).  With a workspace (scatter_workspace_ints
// int32, 16-byte aligned) every token's scale words are staged once and a
// tile kernel writes the tiled scales; with NULL every route's scale words are
// stored into the tiled layout by the scatter kernel itself.
int64_t scatter_workspace_ints(int64_t num_tokens, int64_t total_rows, int64_t E, int64_t K);
cudaError_t launch_quantize_grouped_scatter(const void* x, int64_t num_tokens, int64_t K,
                                            int64_t ldx, const int32_t* dest_rows, int32_t top_k,
                                            int64_t total_rows, const int32_t* offsets, int32_t E,
                                            int32_t* workspace, uint8_t* codes, uint8_t* scales,
                                            int32_t* scale_row_offsets, int32_t* status,
                                            int64_t bound_tiles, bool f16, cudaStream_t stream);

// NVFP4 (16-element blocks, E4M3 scales, device global scale).
cudaError_t launch_quantize_nvfp4(const void* x, int64_t M, int64_t K, int64_t ldx,
                                  const float* global_scale, uint8_t* codes, uint8_t* scales,
                                  bool f16, cudaStream_t stream);
// NVFP4 experts quant: per-segment global scales [E], grouped scale layout.
cudaError_t launch_quantize_nvfp4_grouped(const void* x, int64_t total_rows, int64_t K,
                                          const int32_t* offsets, int32_t E,
                                          const float* global_scales, uint8_t* codes,
                                          uint8_t* scales, int32_t* scale_row_offsets,
                                          int32_t* status, int64_t bound_tiles, bool f16,
                                          cudaStream_t stream);
// NVFP4 experts quant with the dispatch as a scatter (token, route -> row).
// With a workspace (nvfp4_scatter_workspace_ints int32, 16-byte aligned)
// each route's scale bytes are staged by padded row and a tile kernel writes
// the tiled scales; with NULL they go into the tiled layout directly.
int64_t nvfp4_scatter_workspace_ints(int64_t total_rows, int64_t E, int64_t K);
cudaError_t launch_quantize_nvfp4_grouped_scatter(const void* x, int64_t num_tokens, int64_t K,
                                                  int64_t ldx, const int32_t* dest_rows,
                                                  int32_t top_k, int64_t total_rows,
                                                  const int32_t* offsets, int32_t E,
                                                  const float* global_scales, int32_t* workspace,
                                                  uint8_t* codes, uint8_t* scales,
                                                  int32_t* scale_row_offsets, int32_t* status,
                                                  int64_t bound_tiles, bool f16,
                                                  cudaStream_t stream);
cudaError_t launch_dequantize_nvfp4(const uint8_t* codes, const uint8_t* scales,
                                    const float* global_scale, int64_t M, int64_t K, void* y,
                                    cudaStream_t stream);

cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t M, int64_t K,
                              void* y, cudaStream_t stream);

struct SwapArgs {
  const uint8_t* codes_in;
  const uint8_t* scales_in;
  const float* w13_bias_in;
  int32_t E;
  int64_t two_n;
  int64_t K;
  int32_t scales_tiled;
  uint8_t* codes_out;
  uint8_t* scales_out;
  void* w13_bias_out;
  const float* w2_bias_in;
  int64_t w2_bias_numel;
  void* w2_bias_out;
};

cudaError_t launch_swap_w13(const SwapArgs& a, cudaStream_t stream);

// The dispatch permutation from [num_tokens, top_k] expert ids: offsets
// [E+1], dest [num_tokens * top_k] (-1: not dispatched), row_index [rows] or
// NULL, status or NULL; workspace of route_workspace_ints(n, E) int32.
int64_t route_workspace_ints(int64_t n, int64_t E);
cudaError_t launch_moe_route(const int32_t* ids, int64_t num_tokens, int32_t top_k, int32_t E,
                             int32_t* workspace, int32_t* offsets, int32_t* dest,
                             int32_t* row_index, int32_t* status, cudaStream_t stream);

// Number of SMs of the current device (cached per device).
int sm_count();

#ifdef MXFP4_DEBUG_BOUNDS
// Bounds build: out-of-range accesses counted by each translation unit since
// the last read (reading resets the counter).
unsigned int debug_violations_quantize();
unsigned int debug_violations_dispatch();
unsigned int debug_violations_dequantize();
unsigned int debug_violations_nvfp4();
unsigned int debug_violations_swap();
unsigned int debug_violations_route();
#endif

// Launch with programmatic dependent launch allowed: the grid may be
// scheduled while the previous kernel of the stream drains; every kernel of
// this library executes griddepcontrol.wait before touching global memory,
// so it still observes all writes of the preceding work.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned threads, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace mxfp4
