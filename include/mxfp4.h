/*
 * mxfp4.h — C ABI of the GB300 (sm_103a) MXFP4 block-quantization library
 * (libmxfp4_gb300.so).
 *
 * Format (OCP MX, MXFP4): a tensor of BF16 values is cut, along its last
 * dimension K, into blocks of 32 consecutive elements.  Each block gets one
 * E8M0 scale byte s (value 2^(s-127)) and 32 E2M1 codes (4 bits each:
 * sign bit 3, magnitude index bits 2..0 over {0,0.5,1,1.5,2,3,4,6}).
 *
 * Sources (vLLM pull-request summary pages):
 *   [PR43557] "Fix the E8M0 scale computation in the MXFP4 MoE CUTLASS kernel"
 *             (vllm-project/vllm PR #43557): sections "Motivation",
 *             "Implementation breakdown" items 1-3, "Key source snippets"
 *             (compute_reference_e8m0_scale, untile_cutlass_scale and the
 *             cvt_warp_fp16_to_fp4 excerpt), "Risks and impact".
 *   [PR51038] "[Bugfix][Quantization] Fix MXFP4 conversion for FlashInfer
 *             CUTLASS" (PR #51038): "Implementation breakdown" item 2 and the
 *             convert_weight_to_mxfp4_moe_kernel_format / test excerpts.
 *   [PR46915] "Fix the SM90 MXFP4 MoE test weight/scale interleave"
 *             (PR #46915): "Motivation" (packed FP4 weights read through a
 *             FP4->BF16 table).
 *
 * Common conventions of every entry point below
 *   - Kernels run on the calling thread's current CUDA device; every device
 *     pointer must belong to that device (the stream too).
 *   - Every data pointer is DEVICE memory owned by the caller.  The library
 *     never allocates, never frees and never synchronises the host; work is
 *     enqueued on `stream` (a cudaStream_t passed as void*; NULL = the legacy
 *     default stream) and the call returns as soon as it is enqueued.
 *   - Host-checkable errors (shapes, NULL or misaligned pointers, overlapping
 *     input/output ranges) are reported synchronously through the return
 *     value, before anything is enqueued; outputs are then untouched.
 *   - A failed kernel launch returns MXFP4_ECUDA.
 *   - Errors only the device can see (malformed expert offsets, gather
 *     indices or scatter entries out of range) are written to a
 *     caller-provided device status word.
 *   - Size 0 (M == 0, K == 0, E == 0 with no rows) is a valid no-op.
 *   - No kernel of this library waits on another CTA or on the host.
 */
#ifndef MXFP4_GB300_H
#define MXFP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes.  MXFP4_EOFFSETS and MXFP4_EINDEX are only ever written to a
 * device status word. */
typedef enum {
  MXFP4_OK = 0,
  MXFP4_EINVAL = -1,   /* NULL pointer, negative size, bad flag value            */
  MXFP4_EALIGN = -2,   /* pointer or row stride breaks the 16-byte rule            */
  MXFP4_ESHAPE = -3,   /* K % 32 != 0 (16 for NVFP4), ldx < K, odd two_n, overflow */
  MXFP4_EALIAS = -4,   /* an output byte range overlaps an input or another output */
  MXFP4_ECUDA = -5,    /* the CUDA runtime refused a launch                        */
  MXFP4_EOFFSETS = -6, /* device-detected: expert offsets not 0 = o[0] <= ... <= o[E] = rows */
  MXFP4_EINDEX = -7,   /* device-detected: a gather row index outside [0, num_src_rows),
                          or a scatter entry outside [-1, total_rows) */
  MXFP4_ESCRATCH = -8  /* the call needs more scratch than the library's fixed buffer
                          (mxfp4_quantize_grouped_gather_noalloc) */
} mxfp4_status;

/* Bytes of the 128x4-tiled scale buffer of an [M, K] matrix:
 * ceil(M/128)*128 * ceil((K/32)/4)*4.  Every byte of that range is written by
 * the quantizers (pad bytes as 0x00).  Returns 0 when M <= 0, K <= 0,
 * K % 32 != 0 or the byte count would not fit in int64 (sizes no call
 * accepts).  [PR43557] untile_cutlass_scale (padded_M x padded_sK).  Every
 * size query of this header answers 0 in that last case too. */
size_t mxfp4_scale_bytes(int64_t M, int64_t K);

/* Upper bound of the grouped scale buffer for `total_rows` rows split into E
 * segments, each padded to a multiple of 128 rows on its own:
 * floor((total_rows + 127*E)/128) * 128 * ceil((K/32)/4)*4.
 * Returns 0 on invalid arguments. */
size_t mxfp4_grouped_scale_bytes_bound(int64_t total_rows, int32_t E, int64_t K);

/* mxfp4_quantize — BF16 [M, K] -> packed E2M1 codes + tiled E8M0 scales.
 *
 * Defined by [PR43557] "Implementation breakdown" item 1 and the
 * cvt_warp_fp16_to_fp4 excerpt (UE8M0 branch), plus the plain OCP-MX reading
 * of the element step the pages leave implicit:
 *   vecMax = max |x| over the 32-element block;
 *   s = ((bits(vecMax) + 2^21) & 0xFF800000) >> 23 & 0xFF, minus 2 if that
 *       exponent is > 2 else 0, clamped to 254; s = 0 when vecMax <= 0;
 *   code = E2M1 round-to-nearest-even of x * 2^(127-s), saturating at +-6;
 *   every code of a block with s == 0 is 0x0.
 *
 * x       BF16 bits, row r starts at x + r*ldx elements.  16-byte aligned,
 *         ldx % 8 == 0, ldx >= K.  Read only.
 * M, K    rows and columns; K % 32 == 0.
 * codes   [M, K/2] bytes, row stride K/2; byte j of a row holds element 2j
 *         in bits 0..3 and element 2j+1 in bits 4..7.  16-byte aligned.
 * scales  mxfp4_scale_bytes(M, K) bytes, 16-byte aligned, CUTLASS 128x4
 *         tiled layout [ceil(M/128), ceil(K/128), 32, 4, 4]: the scale of row
 *         r, block column c sits at byte
 *           ((r/128)*ceil(K/128) + c/4)*512 + (r%32)*16 + ((r%128)/32)*4 + c%4
 *         ([PR43557] untile_cutlass_scale).  Rows >= M and columns >= K/32
 *         of the padded tile are written as 0x00.
 * Inputs containing Inf or NaN give unspecified codes (but no fault).
 */
int mxfp4_quantize(const void* x, int64_t M, int64_t K, int64_t ldx,
                   uint8_t* codes, uint8_t* scales, void* stream);

/* mxfp4_quantize_f16 — the same method and outputs for IEEE binary16 input.
 * [PR43557] cvt_warp_fp16_to_fp4 excerpt: the kernel converts 16-bit inputs,
 * its block max is a packed half2 max.  The block max is widened to float32
 * exactly and the E8M0 rule applied to its bits; elements are scaled in
 * float32 and rounded to E2M1 as for BF16.  Arguments, layouts, alignment and
 * errors exactly as for mxfp4_quantize (x holds FP16 bit patterns). */
int mxfp4_quantize_f16(const void* x, int64_t M, int64_t K, int64_t ldx,
                       uint8_t* codes, uint8_t* scales, void* stream);

/* mxfp4_quantize_grouped — per-expert ("experts quant") activation quantize.
 *
 * [PR43557] "Implementation breakdown" item 3 (the experts-quant tests) and
 * item 1.  Rows [o[e], o[e+1]) of x form segment e; each segment is quantized
 * exactly as mxfp4_quantize would quantize it alone.  Codes keep the input
 * row order ([total_rows, K/2]).  Segment e's scales form its own tiled,
 * zero-padded buffer of ceil(n_e/128)*128 rows, stored at byte
 * P[e]*ceil(K/128)*4 of `scales`, where P[e] = sum_{e'<e} ceil(n_e'/128)*128.
 *
 * x                  BF16 [total_rows, K], contiguous (row stride K), 16-byte aligned.
 * expert_offsets     DEVICE int32 [E+1]; must satisfy 0 = o[0] <= o[1] <= ...
 *                    <= o[E] = total_rows (checked on the device).
 * codes              [total_rows, K/2], 16-byte aligned.
 * scales             >= mxfp4_grouped_scale_bytes_bound(total_rows, E, K)
 *                    bytes, 16-byte aligned.  Bytes past P[E]*ceil(K/128)*4
 *                    are not touched.
 * scale_row_offsets  DEVICE int32 [E+1], output: P[0..E] (padded row starts).
 * status             DEVICE int32, output, may be NULL: MXFP4_OK, or
 *                    MXFP4_EOFFSETS when the offsets break the rule above;
 *                    in that case scale_row_offsets is filled with -1 and
 *                    codes/scales are left untouched.
 */
int mxfp4_quantize_grouped(const void* x, int64_t total_rows, int64_t K,
                           const int32_t* expert_offsets, int32_t E,
                           uint8_t* codes, uint8_t* scales,
                           int32_t* scale_row_offsets, int32_t* status,
                           void* stream);

/* mxfp4_quantize_grouped_gather — MoE dispatch permutation fused into the
 * grouped quantize: output row r is source row row_index[r] of x.  The result
 * equals mxfp4_quantize_grouped applied to the gathered matrix
 * x[row_index[0..total_rows)], without writing or reading that BF16 matrix.
 * [PR43557] "Implementation breakdown" item 3 (experts quant of the routed,
 * expert-sorted activations).
 *
 * x                  BF16 source rows [num_src_rows, K], row stride ldx
 *                    elements (ldx >= K, ldx % 8 == 0), 16-byte aligned.
 * row_index          DEVICE int32 [total_rows]: source row of every output
 *                    row (e.g. the token of each expert-sorted route).
 * expert_offsets, E, codes, scales, scale_row_offsets: as in
 *                    mxfp4_quantize_grouped, over the total_rows output rows.
 * status             DEVICE int32, output, may be NULL: MXFP4_OK,
 *                    MXFP4_EOFFSETS (as in mxfp4_quantize_grouped), or
 *                    MXFP4_EINDEX when some row_index is outside
 *                    [0, num_src_rows): such rows are quantized as zero rows
 *                    and no out-of-range memory is read.
 *
 * How it runs (the results do not depend on it).  When the inverse map and
 * staged scale words of mxfp4_quantize_grouped_gather_ws fit in the codes of
 * the last quarter of the output rows, the call takes that path and uses
 * those rows of `codes` as its workspace: it clears them, builds the inverse
 * map there, quantizes every source row once into the other rows, then
 * writes the borrowed rows' own codes last, from their source rows.  Until
 * the stream reaches the end of the call, those rows of `codes` hold
 * workspace data.  If the offsets are malformed, the clear is skipped and
 * no code row is written.  Otherwise (small batches) every output row
 * reads its source row itself.
 */
int mxfp4_quantize_grouped_gather(const void* x, int64_t num_src_rows, int64_t K, int64_t ldx,
                                  const int32_t* row_index, int64_t total_rows,
                                  const int32_t* expert_offsets, int32_t E, uint8_t* codes,
                                  uint8_t* scales, int32_t* scale_row_offsets, int32_t* status,
                                  void* stream);

/* mxfp4_quantize_grouped_gather_ws — mxfp4_quantize_grouped_gather with
 * identical results (the same arguments, outputs, status and errors), run
 * through the scatter path: from row_index the library builds its inverse
 * (the rows of every source row) in `workspace`, then reads and quantizes
 * every source row once and writes it to all its rows, instead of reading it
 * once per row (a source row with more than 32 rows is read once more for
 * each row past its 32nd).  [PR43557] "Implementation breakdown" item 3.
 *
 * workspace        DEVICE scratch owned by the caller, 16-byte aligned, at
 *                  least mxfp4_gather_workspace_bytes(num_src_rows, total_rows,
 *                  E, K) bytes, not overlapping any other argument; its
 *                  contents on entry do not matter and on return are
 *                  unspecified.  Two calls in flight at once need two
 *                  workspaces.
 * num_src_rows     <= INT32_MAX / 4.
 * Everything else: as mxfp4_quantize_grouped_gather.  The _f16 form takes
 * IEEE binary16 input.
 *
 * mxfp4_gather_workspace_bytes: the inverse map, 4 * (33T + 1 + 2R) bytes
 * (T = num_src_rows, R = total_rows: a route count and a 32-row bucket per
 * source row, an overflow list of rows past a source row's 32nd), the source
 * row of every padded row, 4 * floor((R + 127E) / 128) * 128 bytes, then,
 * from the next 16-byte
 * boundary, T rows of ceil(K/128) 4-byte scale words, each row padded to a
 * multiple of 4 words: each source row's scale words are stored there once,
 * and a second kernel writes the tiled scales of all rows in whole 512-byte
 * chunks.  0 for negative sizes, K % 32 != 0, num_src_rows > INT32_MAX / 4
 * or R + 127E > INT32_MAX.  With K = 0 it is the inverse map alone, rounded
 * up to 16 bytes.
 */
size_t mxfp4_gather_workspace_bytes(int64_t num_src_rows, int64_t total_rows, int32_t E,
                                    int64_t K);
int mxfp4_quantize_grouped_gather_ws(const void* x, int64_t num_src_rows, int64_t K, int64_t ldx,
                                     const int32_t* row_index, int64_t total_rows,
                                     const int32_t* expert_offsets, int32_t E, void* workspace,
                                     size_t workspace_bytes, uint8_t* codes, uint8_t* scales,
                                     int32_t* scale_row_offsets, int32_t* status, void* stream);
int mxfp4_quantize_grouped_gather_ws_f16(const void* x, int64_t num_src_rows, int64_t K,
                                         int64_t ldx, const int32_t* row_index,
                                         int64_t total_rows, const int32_t* expert_offsets,
                                         int32_t E, void* workspace, size_t workspace_bytes,
                                         uint8_t* codes, uint8_t* scales,
                                         int32_t* scale_row_offsets, int32_t* status,
                                         void* stream);

/* mxfp4_quantize_grouped_gather_noalloc — mxfp4_quantize_grouped_gather_ws
 * without a caller workspace and without any allocation: the inverse map is
 * built in a fixed scratch buffer of MXFP4_NOALLOC_SCRATCH_BYTES inside the
 * library (a device array every GPU that loads the library holds until the
 * process exits).  For callers that cannot allocate device memory.  No
 * counterpart exists in the method's sources.
 *
 * Arguments, outputs and status as mxfp4_quantize_grouped_gather.  Errors are
 * checked in the same order as mxfp4_quantize_grouped_gather_ws (so a shape
 * fault or a size beyond the int32 limits is MXFP4_ESHAPE, a NULL pointer
 * MXFP4_EINVAL); where that call would check the workspace size, this one
 * returns MXFP4_ESCRATCH (before anything is enqueued) when the inverse map
 * alone, mxfp4_gather_workspace_bytes(num_src_rows, total_rows, E, 0),
 * exceeds MXFP4_NOALLOC_SCRATCH_BYTES.  When the whole workspace
 * (mxfp4_gather_workspace_bytes(num_src_rows, total_rows, E, K)) fits, the
 * call runs exactly as mxfp4_quantize_grouped_gather_ws; otherwise the
 * scatter stores every row's scale words into the tiled layout itself (same
 * results, slower).
 * Every call shares the one buffer of its device: two calls that can overlap
 * on the GPU (different streams, or a graph replayed concurrently) race and
 * give wrong results; serialise them.  The buffer keeps the last call's
 * contents; each call clears what must start at zero.  A call looks up the
 * buffer's device address (a host-side query) on its device's first call
 * and again when the current context has changed since (after
 * cudaDeviceReset the buffer lives at a new address): make the first call
 * on a device, and the first after a reset, outside any stream capture.
 */
#define MXFP4_NOALLOC_SCRATCH_BYTES (4u << 20)
int mxfp4_quantize_grouped_gather_noalloc(const void* x, int64_t num_src_rows, int64_t K,
                                          int64_t ldx, const int32_t* row_index,
                                          int64_t total_rows, const int32_t* expert_offsets,
                                          int32_t E, uint8_t* codes, uint8_t* scales,
                                          int32_t* scale_row_offsets, int32_t* status,
                                          void* stream);

/* mxfp4_quantize_grouped_scatter — the same dispatch given in the direction
 * a router's sort produces it (token, route -> row): each token row of x is
 * read and quantized once, and its codes and scale bytes are written to every
 * row its routes land on.  Where every row 0..total_rows-1 is targeted
 * exactly once, the result equals mxfp4_quantize_grouped_gather with the
 * inverse map.  [PR43557] "Implementation breakdown" item 3 (experts quant of
 * the routed, expert-sorted activations).
 *
 * x                  BF16 token rows [num_tokens, K], row stride ldx elements
 *                    (ldx >= K, ldx % 8 == 0), 16-byte aligned.
 * dest_rows          DEVICE int32 [num_tokens, top_k], row-major: the row of
 *                    the expert-sorted batch that route j of token t lands
 *                    on, or -1 for a route that is not dispatched.
 *                    1 <= top_k <= MXFP4_SCATTER_MAX_TOP_K.  No row may be
 *                    the target of two different tokens (that row's bytes
 *                    would be unspecified).
 * expert_offsets, E, codes, scales, scale_row_offsets: as in
 *                    mxfp4_quantize_grouped, over the total_rows rows of the
 *                    expert-sorted batch.  Rows that no route targets are not
 *                    written (neither their codes nor their scale bytes); the
 *                    pad rows of every segment get zero scale bytes.
 * status             DEVICE int32, output, may be NULL: MXFP4_OK,
 *                    MXFP4_EOFFSETS (as in mxfp4_quantize_grouped, nothing
 *                    else written), or MXFP4_EINDEX when some entry is
 *                    outside [-1, total_rows): such entries are skipped.
 */
#define MXFP4_SCATTER_MAX_TOP_K 32
int mxfp4_quantize_grouped_scatter(const void* x, int64_t num_tokens, int64_t K, int64_t ldx,
                                   const int32_t* dest_rows, int32_t top_k, int64_t total_rows,
                                   const int32_t* expert_offsets, int32_t E, uint8_t* codes,
                                   uint8_t* scales, int32_t* scale_row_offsets,
                                   int32_t* status, void* stream);

/* mxfp4_quantize_grouped_scatter_ws — mxfp4_quantize_grouped_scatter with
 * identical results (the same arguments, outputs, status and errors; rows
 * that no route targets keep their codes and their scale bytes) and a
 * caller-provided workspace: the scatter kernel stores each token's scale
 * words once into the workspace instead of every route's words into the
 * tiled layout, then a second kernel writes the tiled scales in whole
 * 512-byte chunks (an untargeted row's scale bytes are read back and written
 * unchanged).
 *
 * workspace        DEVICE scratch owned by the caller, 16-byte aligned, at
 *                  least mxfp4_scatter_workspace_bytes(num_tokens,
 *                  total_rows, E, K) bytes, not overlapping any other
 *                  argument; its contents on entry do not matter and on
 *                  return are unspecified.  Two calls in flight at once need
 *                  two workspaces.
 * num_tokens       <= INT32_MAX / 4.
 * The _f16 form takes IEEE binary16 input.
 *
 * mxfp4_scatter_workspace_bytes: 4 * floor((R + 127E) / 128) * 128 bytes
 * (the token of every padded row, R = total_rows) plus num_tokens rows of
 * ceil(K/128) 4-byte scale words, each row padded to a multiple of 4 words;
 * 0 for negative sizes, K % 32 != 0, num_tokens > INT32_MAX / 4 or
 * R + 127E > INT32_MAX.
 */
size_t mxfp4_scatter_workspace_bytes(int64_t num_tokens, int64_t total_rows, int32_t E,
                                     int64_t K);
int mxfp4_quantize_grouped_scatter_ws(const void* x, int64_t num_tokens, int64_t K, int64_t ldx,
                                      const int32_t* dest_rows, int32_t top_k,
                                      int64_t total_rows, const int32_t* expert_offsets,
                                      int32_t E, void* workspace, size_t workspace_bytes,
                                      uint8_t* codes, uint8_t* scales,
                                      int32_t* scale_row_offsets, int32_t* status,
                                      void* stream);
int mxfp4_quantize_grouped_scatter_ws_f16(const void* x, int64_t num_tokens, int64_t K,
                                          int64_t ldx, const int32_t* dest_rows, int32_t top_k,
                                          int64_t total_rows, const int32_t* expert_offsets,
                                          int32_t E, void* workspace, size_t workspace_bytes,
                                          uint8_t* codes, uint8_t* scales,
                                          int32_t* scale_row_offsets, int32_t* status,
                                          void* stream);

/* FP16 input for the grouped forms: mxfp4_quantize_grouped_f16,
 * mxfp4_quantize_grouped_gather_f16 and mxfp4_quantize_grouped_scatter_f16
 * take IEEE binary16 bit patterns in x and otherwise behave exactly as the
 * BF16 calls of the same name (arguments, layouts, status, errors), with the
 * element step of mxfp4_quantize_f16 ([PR43557] cvt_warp_fp16_to_fp4: the
 * experts-quant kernel converts 16-bit inputs of either kind). */
int mxfp4_quantize_grouped_f16(const void* x, int64_t total_rows, int64_t K,
                               const int32_t* expert_offsets, int32_t E,
                               uint8_t* codes, uint8_t* scales,
                               int32_t* scale_row_offsets, int32_t* status,
                               void* stream);
int mxfp4_quantize_grouped_gather_f16(const void* x, int64_t num_src_rows, int64_t K, int64_t ldx,
                                      const int32_t* row_index, int64_t total_rows,
                                      const int32_t* expert_offsets, int32_t E, uint8_t* codes,
                                      uint8_t* scales, int32_t* scale_row_offsets,
                                      int32_t* status, void* stream);
int mxfp4_quantize_grouped_scatter_f16(const void* x, int64_t num_tokens, int64_t K, int64_t ldx,
                                       const int32_t* dest_rows, int32_t top_k,
                                       int64_t total_rows, const int32_t* expert_offsets,
                                       int32_t E, uint8_t* codes, uint8_t* scales,
                                       int32_t* scale_row_offsets, int32_t* status,
                                       void* stream);

/* mxfp4_dequantize — packed codes + tiled scales -> BF16 [M, K].
 *
 * The inverse mapping of the format ([PR46915] "Motivation": FP4 -> BF16
 * table; [PR43557] cvt_warp_fp16_to_fp4 excerpt: scale value 2^(s-127)):
 *   y = BF16_RNE(e2m1(code) * 2^(s-127)); overflow gives +-Inf, code 0x8
 *   gives -0.0, s == 255 (E8M0 NaN) gives 0x7FC0 for the whole block.
 *
 * codes   [M, K/2], layout as written by mxfp4_quantize, 16-byte aligned.
 * scales  mxfp4_scale_bytes(M, K) bytes, tiled layout, 16-byte aligned.
 * y       BF16 [M, K], contiguous, 16-byte aligned, written.
 */
int mxfp4_dequantize(const uint8_t* codes, const uint8_t* scales,
                     int64_t M, int64_t K, void* y, void* stream);

/* mxfp4_swap_w13 — fused gate/up weights [w1; w3] -> [w3; w1].
 *
 * [PR51038] "Implementation breakdown" item 2 and the
 * convert_weight_to_mxfp4_moe_kernel_format branch / its test: per expert,
 * rows [0, N) and [N, 2N) of the w13 codes and scales change places
 * (out row r = in row (r + N) mod 2N); the w13 bias halves change places the
 * same way and are cast FP32 -> BF16 (RNE); the w2 bias is only cast.
 *
 * codes_in/out   [E, two_n, K/2] bytes, 16-byte aligned.
 * scales_in/out  scales_tiled == 0: flat [E, two_n, K/32] bytes;
 *                scales_tiled == 1: E consecutive tiled buffers of
 *                mxfp4_scale_bytes(two_n, K) bytes each (rows are swapped by
 *                logical row; pad bytes are written 0x00).  16-byte aligned.
 * w13_bias_in    FP32 [E, two_n] or NULL (then w13_bias_out is ignored).
 * w13_bias_out   BF16 [E, two_n].
 * w2_bias_in     FP32 [w2_bias_numel] or NULL (then w2_bias_out is ignored).
 * w2_bias_out    BF16 [w2_bias_numel].
 * two_n must be even, K % 32 == 0.  Out-of-place only (MXFP4_EALIAS if any
 * output range overlaps an input range).
 */
int mxfp4_swap_w13(const uint8_t* codes_in, const uint8_t* scales_in,
                   const float* w13_bias_in, int32_t E, int64_t two_n, int64_t K,
                   int32_t scales_tiled, uint8_t* codes_out, uint8_t* scales_out,
                   void* w13_bias_out, const float* w2_bias_in,
                   int64_t w2_bias_numel, void* w2_bias_out, void* stream);

/* mxfp4_nvfp4_grouped_scale_bytes_bound — scale buffer size that always
 * suffices for mxfp4_quantize_nvfp4_grouped:
 * floor((total_rows + 127*E) / 128) * 128 * ceil(K/64) * 4 bytes
 * (0 for invalid sizes). */
size_t mxfp4_nvfp4_grouped_scale_bytes_bound(int64_t total_rows, int32_t E, int64_t K);

/* mxfp4_quantize_nvfp4_grouped — NVFP4 "experts quant": the NVFP4 branch of
 * the experts-quant kernel ([PR43557] "Implementation breakdown" items 1 and
 * 3) over expert segments.  Rows [o[e], o[e+1]) of x form segment e; each
 * segment is quantized exactly as mxfp4_quantize_nvfp4 would quantize it
 * alone with global scale global_scales[e].  Codes keep the row order;
 * segment e's tiled E4M3 scales (16-element columns, padded to 128 rows)
 * start at byte P[e] * ceil(K/64) * 4, P[e] = sum_{e'<e} ceil(n_e'/128)*128.
 * One global scale per expert is this library's reading (the pages show the
 * scale as one argument of the conversion); a single scale for all experts
 * is the case of E equal entries.
 *
 * x                  BF16 [total_rows, K], contiguous, 16-byte aligned; K % 16 == 0.
 * expert_offsets     DEVICE int32 [E+1], 0 = o[0] <= ... <= o[E] = total_rows
 *                    (checked on the device).
 * global_scales      DEVICE float32 [E], positive finite (not checked); below
 *                    2^119 for fully specified results, as mxfp4_quantize_nvfp4.
 * codes              [total_rows, K/2]; scales >= the bound above, 16-byte
 *                    aligned; bytes past P[E] * ceil(K/64) * 4 are not touched.
 * scale_row_offsets  DEVICE int32 [E+1], output P[0..E].
 * status             DEVICE int32, output, may be NULL: MXFP4_OK or
 *                    MXFP4_EOFFSETS (then scale_row_offsets is all -1 and
 *                    codes/scales are left untouched).
 */
int mxfp4_quantize_nvfp4_grouped(const void* x, int64_t total_rows, int64_t K,
                                 const int32_t* expert_offsets, int32_t E,
                                 const float* global_scales, uint8_t* codes, uint8_t* scales,
                                 int32_t* scale_row_offsets, int32_t* status, void* stream);
/* The same experts quant for IEEE binary16 input (x holds FP16 bit patterns;
 * everything else as mxfp4_quantize_nvfp4_grouped, element step as
 * mxfp4_quantize_nvfp4_f16). */
int mxfp4_quantize_nvfp4_grouped_f16(const void* x, int64_t total_rows, int64_t K,
                                     const int32_t* expert_offsets, int32_t E,
                                     const float* global_scales, uint8_t* codes,
                                     uint8_t* scales, int32_t* scale_row_offsets,
                                     int32_t* status, void* stream);

/* mxfp4_quantize_nvfp4_grouped_scatter — the NVFP4 experts quant with the
 * MoE dispatch fused in as a scatter: route j of token t lands on row
 * dest_rows[t][j] of the expert-sorted batch (-1: not dispatched).  Each
 * token row is read once and its block maxima taken once; each route's codes
 * and E4M3 scales use the global scale of the segment its row falls in, so
 * the result equals mxfp4_quantize_nvfp4_grouped of the batch the routes
 * fill.  [PR43557] "Implementation breakdown" items 1 and 3 (the NVFP4 branch
 * of the experts quant of the routed activations).
 *
 * x, dest_rows, top_k, total_rows, expert_offsets, E, status: as in
 * mxfp4_quantize_grouped_scatter (rows no route targets are not written; pad
 * rows get zero scale bytes; entries outside [-1, total_rows) are skipped and
 * reported as MXFP4_EINDEX; no row may be the target of two tokens), with
 * K % 16 == 0.
 * global_scales, codes, scales, scale_row_offsets: as in
 * mxfp4_quantize_nvfp4_grouped (scales >= mxfp4_nvfp4_grouped_scale_bytes_bound).
 * The _f16 form takes IEEE binary16 input.
 */
int mxfp4_quantize_nvfp4_grouped_scatter(const void* x, int64_t num_tokens, int64_t K,
                                         int64_t ldx, const int32_t* dest_rows, int32_t top_k,
                                         int64_t total_rows, const int32_t* expert_offsets,
                                         int32_t E, const float* global_scales, uint8_t* codes,
                                         uint8_t* scales, int32_t* scale_row_offsets,
                                         int32_t* status, void* stream);
int mxfp4_quantize_nvfp4_grouped_scatter_f16(const void* x, int64_t num_tokens, int64_t K,
                                             int64_t ldx, const int32_t* dest_rows,
                                             int32_t top_k, int64_t total_rows,
                                             const int32_t* expert_offsets, int32_t E,
                                             const float* global_scales, uint8_t* codes,
                                             uint8_t* scales, int32_t* scale_row_offsets,
                                             int32_t* status, void* stream);

/* mxfp4_quantize_nvfp4_grouped_scatter_ws — the same call with identical
 * results (rows no route targets keep their codes and scale bytes) and a
 * caller-provided workspace: each route's scale bytes are stored as one
 * contiguous row of the workspace (indexed by the route's padded row) instead
 * of as 4-byte words scattered over the tiled layout, and a second kernel
 * writes the tiled scales in whole 512-byte chunks.  A token whose routes all
 * land in experts of one global scale (the same bits) has the same scale
 * bytes on every route; it stores them once, in its first route's row.
 *
 * workspace        DEVICE scratch owned by the caller, 16-byte aligned, at
 *                  least mxfp4_nvfp4_scatter_workspace_bytes(total_rows, E, K)
 *                  bytes, not overlapping any other argument; contents on
 *                  entry do not matter, on return unspecified.
 *
 * mxfp4_nvfp4_scatter_workspace_bytes: PT * (4 + 4 * ceil4(ceil(K/64)))
 * bytes, PT = floor((total_rows + 127E) / 128) * 128 padded rows (for every
 * padded row the staged row its scale bytes are read from, then one staged
 * scale row per padded row); 0 for
 * negative sizes, K % 16 != 0 or total_rows + 127E > INT32_MAX.
 */
size_t mxfp4_nvfp4_scatter_workspace_bytes(int64_t total_rows, int32_t E, int64_t K);
int mxfp4_quantize_nvfp4_grouped_scatter_ws(const void* x, int64_t num_tokens, int64_t K,
                                            int64_t ldx, const int32_t* dest_rows, int32_t top_k,
                                            int64_t total_rows, const int32_t* expert_offsets,
                                            int32_t E, const float* global_scales,
                                            void* workspace, size_t workspace_bytes,
                                            uint8_t* codes, uint8_t* scales,
                                            int32_t* scale_row_offsets, int32_t* status,
                                            void* stream);
int mxfp4_quantize_nvfp4_grouped_scatter_ws_f16(const void* x, int64_t num_tokens, int64_t K,
                                                int64_t ldx, const int32_t* dest_rows,
                                                int32_t top_k, int64_t total_rows,
                                                const int32_t* expert_offsets, int32_t E,
                                                const float* global_scales, void* workspace,
                                                size_t workspace_bytes, uint8_t* codes,
                                                uint8_t* scales, int32_t* scale_row_offsets,
                                                int32_t* status, void* stream);

/* mxfp4_moe_route — the dispatch permutation the grouped, scatter and
 * gather calls take, from the router's choices ([PR43557] "Implementation
 * breakdown" item 3: the experts quant takes the routed activations sorted
 * by expert; this is that sort, on the device).
 *
 * topk_ids        DEVICE int32 [num_tokens, top_k]: the expert of route j of
 *                 token t at t * top_k + j; -1: the route is not dispatched.
 * num_tokens      >= 0; top_k >= 1; num_tokens * top_k <= INT32_MAX / 2.
 * E               1 <= E <= MXFP4_ROUTE_MAX_EXPERTS.
 * workspace       DEVICE, >= mxfp4_route_workspace_bytes(num_tokens, top_k, E)
 *                 bytes, 16-byte aligned, contents on entry irrelevant
 *                 (NULL allowed when num_tokens * top_k == 0).
 * expert_offsets  DEVICE int32 [E+1], out: the first row of every expert and
 *                 the number of rows (the expert_offsets of the grouped calls).
 * dest_rows       DEVICE int32 [num_tokens, top_k], out: the row of every
 *                 route, -1 when not dispatched (the scatter calls' dest_rows).
 * row_index       DEVICE int32 [num_tokens * top_k] or NULL, out: the token of
 *                 every row; entries from expert_offsets[E] on are not written
 *                 (the gather calls' row_index).
 * status          DEVICE int32 or NULL, out: MXFP4_OK, or MXFP4_EINDEX when
 *                 an id is neither -1 nor in [0, E) (that route is dropped).
 * Rows are the dispatched routes in order of expert, then of t * top_k + j:
 * deterministic, and in token order within every expert.  Errors (returned
 * before anything is enqueued): MXFP4_EINVAL for negative sizes, top_k < 1,
 * E < 1, a NULL pointer or a small workspace; MXFP4_ESHAPE for E or the
 * number of routes above the limits; MXFP4_EALIGN for an int32 array not
 * 4-byte or a workspace not 16-byte aligned; MXFP4_EALIAS for overlapping
 * buffers; MXFP4_ECUDA for a refused launch.  Asynchronous on `stream`. */
#define MXFP4_ROUTE_MAX_EXPERTS 8192
size_t mxfp4_route_workspace_bytes(int64_t num_tokens, int32_t top_k, int32_t E);
int mxfp4_moe_route(const int32_t* topk_ids, int64_t num_tokens, int32_t top_k, int32_t E,
                    void* workspace, size_t workspace_bytes, int32_t* expert_offsets,
                    int32_t* dest_rows, int32_t* row_index, int32_t* status, void* stream);

/* ---------------------------------------------------------------- NVFP4
 * The other branch of the same quantize kernel on [PR43557] ("Implementation
 * breakdown" item 1, the non-UE8M0 branch of the cvt_warp_fp16_to_fp4
 * excerpt, and "Review highlights"): one FP8 E4M3 scale per block,
 * SFScaleVal * vecMax / 6, and the elements scaled with the E4M3-rounded
 * value so quantize and dequantize agree.  Readings where the page is
 * silent: 16-element blocks; every step one IEEE float32 operation rounded
 * to nearest even:
 *   q = vecMax / 6; sf = g * q; byte = E4M3_RNE_satfinite(sf);
 *   inv = g / float(byte); code = E2M1_RNE_saturating(x * inv);
 *   blocks whose byte is 0 emit zero codes;
 *   dequantize: y = BF16_RNE((e2m1(code) * float(byte)) * (1 / g)), and
 *   0x7FC0 (the BF16 NaN) for every element of a block whose scale byte is
 *   the E4M3 NaN (0x7F or 0xFF); specified for g >= 2^-127 (1 / g finite).
 * g is the per-tensor global scale (SFScaleVal), a positive finite float
 * read from DEVICE memory (global_scale, 4-byte aligned).  The results are
 * specified for g < 2^119, where g / float(byte) stays finite for every
 * nonzero byte (the smallest is 2^-9).  Above it a block with a small byte
 * has inv = +inf, its zero elements give 0 * inf = NaN, and their codes are
 * unspecified (E2M1 has no NaN; the sequence above does not say how one is
 * encoded); every other output is as above.  A caller's 448 * 6 / amax
 * exceeds 2^119 only for amax below 4e-33.
 * Scales use the 128x4 tiled layout of mxfp4_quantize over K/16 scale
 * columns: mxfp4_nvfp4_scale_bytes(M, K) = ceil(M/128)*128 * ceil(K/64)*4
 * bytes, pad bytes 0x00.  Codes: [M, K/2], element 2j in the low nibble.
 * K % 16 == 0; other arguments, alignment and errors as mxfp4_quantize /
 * mxfp4_dequantize. */
size_t mxfp4_nvfp4_scale_bytes(int64_t M, int64_t K);
int mxfp4_quantize_nvfp4(const void* x, int64_t M, int64_t K, int64_t ldx,
                         const float* global_scale, uint8_t* codes, uint8_t* scales,
                         void* stream);
/* mxfp4_quantize_nvfp4_f16 — NVFP4 of IEEE binary16 input ([PR43557]
 * cvt_warp_fp16_to_fp4 takes either 16-bit type on both branches).  The
 * block max is a packed half2 max widened to float32 exactly; every later
 * step is the float32 sequence above.  Arguments, layouts, alignment and
 * errors exactly as mxfp4_quantize_nvfp4 (x holds FP16 bit patterns). */
int mxfp4_quantize_nvfp4_f16(const void* x, int64_t M, int64_t K, int64_t ldx,
                             const float* global_scale, uint8_t* codes, uint8_t* scales,
                             void* stream);
int mxfp4_dequantize_nvfp4(const uint8_t* codes, const uint8_t* scales,
                           const float* global_scale, int64_t M, int64_t K, void* y,
                           void* stream);

/* Static, NUL-terminated description of a status code (never NULL). */
const char* mxfp4_status_string(int status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int mxfp4_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_GB300_H */
