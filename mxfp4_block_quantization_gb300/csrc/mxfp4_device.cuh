// mxfp4_device.cuh — device-side building blocks of the sm_103a MXFP4 kernels.
//
// Format sources (vLLM pull-request summary pages):
//   [PR43557] "Fix the E8M0 scale computation in the MXFP4 MoE CUTLASS kernel":
//             "Implementation breakdown" item 1 and the cvt_warp_fp16_to_fp4
//             excerpt (E8M0 scale rule, scale value 2^(s-127)); the
//             untile_cutlass_scale snippet (128x4 tiled scale layout).
//   OCP MX v1.0 for the E2M1 element encoding the pages leave implicit.
#pragma once

#include <cstdint>

namespace mxfp4 {

// ---------------------------------------------------------------- geometry
constexpr int kBlock = 32;          // elements per scale block
constexpr int kTileRows = 128;      // rows of one tiled scale chunk
constexpr int kTileBlocks = 4;      // scale columns of one tiled scale chunk
constexpr int kTileCols = kTileBlocks * kBlock;   // 128 BF16 columns
constexpr int kChunkBytes = kTileRows * kTileBlocks;  // 512 B of scales per tile

// Byte offset of (local row lr in [0,128), block b in [0,4)) inside one 512 B
// tiled chunk: [32 outerM][4 innerM][4 innerK] with outerM = lr % 32,
// innerM = lr / 32 ([PR43557] untile_cutlass_scale permutation).
__device__ __forceinline__ int chunk_offset(int lr, int b) {
  return (lr & 31) * 16 + (lr >> 5) * 4 + b;
}

// ------------------------------------------------------------ E8M0 scale
// [PR43557] UE8M0 branch: add 2^21 to the float bits of vecMax (rounds the
// exponent up when the mantissa is >= 0.75), take the exponent field,
// subtract 2 when it is > 2 (else 0), cap at 254.  vecMax arrives as the
// BF16 bit pattern of a non-negative value (sign already cleared), i.e. the
// float bits are m << 16, so the add is (m + 0x20) on the BF16 pattern and
// the 8-bit exponent field is bits 7..14 of that sum (bit 15 set only by the
// NaN patterns >= 0x7FE0, where the 32-bit form wraps the same way).
__device__ __forceinline__ uint32_t e8m0_from_absmax_bf16(uint32_t m) {
  uint32_t e = ((m + 0x20u) >> 7) & 0xFFu;
  uint32_t s = e > 2u ? e - 2u : 0u;
  return s < 254u ? s : 254u;
}

// The same rule on the float32 bits of a non-negative vecMax (used for FP16
// input, whose block max is first widened to float32 exactly).
__device__ __forceinline__ uint32_t e8m0_from_absmax_f32bits(uint32_t bits) {
  uint32_t e = ((bits + (1u << 21)) & 0xFF800000u) >> 23 & 0xFFu;
  uint32_t s = e > 2u ? e - 2u : 0u;
  return s < 254u ? s : 254u;
}

// 2^(127 - s) as float bits for s in [1, 253]: biased exponent 254 - s.
__device__ __forceinline__ float inv_scale_from_e8m0(uint32_t s) {
  return __uint_as_float((254u - s) << 23);
}

// 2^(s - 127) as a float, every s in [0, 254]: s == 0 is the subnormal
// 2^-127 (mantissa bit 22).  s == 255 (E8M0 NaN) is handled by the caller.
__device__ __forceinline__ float scale_from_e8m0(uint32_t s) {
  return __uint_as_float(s ? (s << 23) : 0x00400000u);
}

// ------------------------------------------------- E2M1 conversion (PTX)
// Two float32 -> one byte of two E2M1 codes, round to nearest even with
// saturation to +-6 (sm_100-family instruction).  `lo` lands in bits 0..3,
// `hi` in bits 4..7.  Four such bytes are packed into one 32-bit word,
// element 2j in the low nibble of byte j.
__device__ __forceinline__ uint32_t cvt_e2m1x8(float a0, float a1, float a2, float a3,
                                               float a4, float a5, float a6, float a7) {
  uint32_t r;
  asm("{\n\t"
      ".reg .b8 q0, q1, q2, q3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t"
      "}"
      : "=r"(r)
      : "f"(a0), "f"(a1), "f"(a2), "f"(a3), "f"(a4), "f"(a5), "f"(a6), "f"(a7));
  return r;
}

// Four packed BF16x2 words (elements 0..7, element 0 in the low half of w0)
// times a power of two `f` -> one 32-bit word of eight E2M1 codes (element
// 2j in the low nibble of byte j), via float32 pairs and the packed f32x2
// multiply.  Exact: a BF16 value times 2^k stays representable in float32
// (results below 2^-126 may round, towards +-0, far below the first E2M1
// rounding threshold 0.25).
__device__ __forceinline__ uint32_t scale_cvt_e2m1x8(uint4 w, float f) {
  uint32_t r;
  asm("{\n\t"
      ".reg .b64 p0, p1, p2, p3, fs;\n\t"
      ".reg .b32 l0, h0, l1, h1, l2, h2, l3, h3;\n\t"
      ".reg .b8 q0, q1, q2, q3;\n\t"
      "shl.b32 l0, %1, 16;\n\t"
      "and.b32 h0, %1, 0xFFFF0000;\n\t"
      "shl.b32 l1, %2, 16;\n\t"
      "and.b32 h1, %2, 0xFFFF0000;\n\t"
      "shl.b32 l2, %3, 16;\n\t"
      "and.b32 h2, %3, 0xFFFF0000;\n\t"
      "shl.b32 l3, %4, 16;\n\t"
      "and.b32 h3, %4, 0xFFFF0000;\n\t"
      "mov.b64 fs, {%5, %5};\n\t"
      "mov.b64 p0, {l0, h0};\n\t"
      "mov.b64 p1, {l1, h1};\n\t"
      "mov.b64 p2, {l2, h2};\n\t"
      "mov.b64 p3, {l3, h3};\n\t"
      "mul.rn.f32x2 p0, p0, fs;\n\t"
      "mul.rn.f32x2 p1, p1, fs;\n\t"
      "mul.rn.f32x2 p2, p2, fs;\n\t"
      "mul.rn.f32x2 p3, p3, fs;\n\t"
      "mov.b64 {l0, h0}, p0;\n\t"
      "mov.b64 {l1, h1}, p1;\n\t"
      "mov.b64 {l2, h2}, p2;\n\t"
      "mov.b64 {l3, h3}, p3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, h0, l0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, h1, l1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, h2, l2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, h3, l3;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t"
      "}"
      : "=r"(r)
      : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "f"(f));
  return r;
}

// The FP16 counterpart: four packed F16x2 words -> one word of eight E2M1
// codes; each half is widened to float32 exactly (cvt.f32.f16) before the
// power-of-two scaling.
__device__ __forceinline__ uint32_t scale_cvt_e2m1x8_f16(uint4 w, float f) {
  uint32_t r;
  asm("{\n\t"
      ".reg .b64 p0, p1, p2, p3, fs;\n\t"
      ".reg .b16 a0, b0, a1, b1, a2, b2, a3, b3;\n\t"
      ".reg .f32 l0, h0, l1, h1, l2, h2, l3, h3;\n\t"
      ".reg .b8 q0, q1, q2, q3;\n\t"
      "mov.b32 {a0, b0}, %1;\n\t"
      "mov.b32 {a1, b1}, %2;\n\t"
      "mov.b32 {a2, b2}, %3;\n\t"
      "mov.b32 {a3, b3}, %4;\n\t"
      "cvt.f32.f16 l0, a0;\n\t"
      "cvt.f32.f16 h0, b0;\n\t"
      "cvt.f32.f16 l1, a1;\n\t"
      "cvt.f32.f16 h1, b1;\n\t"
      "cvt.f32.f16 l2, a2;\n\t"
      "cvt.f32.f16 h2, b2;\n\t"
      "cvt.f32.f16 l3, a3;\n\t"
      "cvt.f32.f16 h3, b3;\n\t"
      "mov.b64 fs, {%5, %5};\n\t"
      "mov.b64 p0, {l0, h0};\n\t"
      "mov.b64 p1, {l1, h1};\n\t"
      "mov.b64 p2, {l2, h2};\n\t"
      "mov.b64 p3, {l3, h3};\n\t"
      "mul.rn.f32x2 p0, p0, fs;\n\t"
      "mul.rn.f32x2 p1, p1, fs;\n\t"
      "mul.rn.f32x2 p2, p2, fs;\n\t"
      "mul.rn.f32x2 p3, p3, fs;\n\t"
      "mov.b64 {l0, h0}, p0;\n\t"
      "mov.b64 {l1, h1}, p1;\n\t"
      "mov.b64 {l2, h2}, p2;\n\t"
      "mov.b64 {l3, h3}, p3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q0, h0, l0;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q1, h1, l1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q2, h2, l2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 q3, h3, l3;\n\t"
      "mov.b32 %0, {q0, q1, q2, q3};\n\t"
      "}"
      : "=r"(r)
      : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "f"(f));
  return r;
}

// One byte of two E2M1 codes -> two halves (f16x2), low nibble in the low half.
__device__ __forceinline__ uint32_t cvt_e2m1x2_to_f16x2(uint32_t byte_in_low_bits) {
  uint32_t r;
  uint16_t v = static_cast<uint16_t>(byte_in_low_bits);
  asm("{\n\t"
      ".reg .b8 lo, hi;\n\t"
      "mov.b16 {lo, hi}, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, lo;\n\t"
      "}"
      : "=r"(r)
      : "h"(v));
  return r;
}

// Two float32 -> BF16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float half_lo_to_f32(uint32_t h2) {
  float f;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, l;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}
__device__ __forceinline__ float half_hi_to_f32(uint32_t h2) {
  float f;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, h;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}

// ------------------------------------------------ FP8 E4M3 (NVFP4 scales)
// float32 -> E4M3 byte, round to nearest even, saturating at +-448.
__device__ __forceinline__ uint32_t cvt_e4m3_satfinite(float f) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(f));
  return r & 0xFFu;
}

// E4M3 byte -> float32 (exact, through f16).
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  uint32_t h2;
  const uint16_t v = static_cast<uint16_t>(byte);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  return half_lo_to_f32(h2);
}

// -------------------------------------------------------- memory access
// Streaming 16-byte load of data read exactly once: read-only path, no L1
// allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 32-byte load (two uint4); the address must be 32-byte aligned.
__device__ __forceinline__ void ld_stream_v8(const void* p, uint4& a, uint4& b) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z),
                 "=r"(b.w)
               : "l"(p));
}

__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Streaming stores (evict-first: outputs are not re-read by this kernel).
__device__ __forceinline__ void st_stream_u32(void* p, uint32_t v) {
  asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_stream_v2(void* p, uint2 v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}
// 32-byte store (two uint4); the address must be 32-byte aligned.
__device__ __forceinline__ void st_stream_v8(void* p, uint4 a, uint4 b) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a.x),
               "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}
__device__ __forceinline__ void st_stream_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Per-half max of |a| and |b| for BF16x2 (the sign bit of each half becomes
// the xor of the input signs and is cleared by the caller).
__device__ __forceinline__ uint32_t max_abs_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t max_abs_f16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// FP16 bit pattern (low 16 bits) -> float32 bits, exact.
__device__ __forceinline__ uint32_t f16_bits_to_f32_bits(uint32_t h) {
  float f;
  const uint16_t v = static_cast<uint16_t>(h);
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"(v));
  return __float_as_uint(f);
}

// ------------------------------------------------- bounds-checking build
// Compiled with -DMXFP4_DEBUG_BOUNDS (libmxfp4_gb300_debug.so), every global
// load and store of every kernel is first checked against the byte range of
// the buffer it belongs to, as the host derived it from the call's
// arguments.  An access outside its range is skipped (a skipped load yields
// zeros) and counted in a per-translation-unit device counter; nothing
// traps.  In the normal build the checks compile away.
// 256-bit loads need every lane address 32-byte aligned: the base and the
// row stride (the column offsets are multiples of 32 bytes).
inline bool vec32_ok(const void* x, int64_t ldx_bytes) {
  return (reinterpret_cast<uintptr_t>(x) % 32 == 0) && (ldx_bytes % 32 == 0);
}

struct DebugRanges {
  uintptr_t lo[8];
  uintptr_t hi[8];
};

#ifdef MXFP4_DEBUG_BOUNDS
static __device__ unsigned int g_debug_violations;

__device__ __forceinline__ bool debug_in_bounds(const DebugRanges& r, int slot, const void* p,
                                                unsigned bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const bool ok = a >= r.lo[slot] && a + bytes <= r.hi[slot];
  if (!ok) atomicAdd(&g_debug_violations, 1u);
  return ok;
}
#define MXFP4_IN_BOUNDS(params, slot, ptr, bytes) \
  ::mxfp4::debug_in_bounds((params).dbg, (slot), (ptr), (bytes))
#else
#define MXFP4_IN_BOUNDS(params, slot, ptr, bytes) true
#endif

inline void debug_range(DebugRanges& r, int slot, const void* p, int64_t bytes) {
  r.lo[slot] = reinterpret_cast<uintptr_t>(p);
  r.hi[slot] = r.lo[slot] + static_cast<uintptr_t>(bytes > 0 ? bytes : 0);
}

// ------------------------------------------- one lane's 16 elements
// The quantize kernels give each lane 16 consecutive elements of a row (one
// 32-byte load, or two 16-byte loads when the input is only 16-byte
// aligned); two neighbouring lanes form one 32-element block.
constexpr int kElems = 16;                                  // elements per lane per pass
constexpr int kLanesPerRow = kTileCols / kElems;            // 8 lanes cover 128 columns

// One lane's 16 BF16 elements (32 bytes) of one row.
template <bool kVec32>
__device__ __forceinline__ void load32(const uint8_t* src, uint4 (&v)[2]) {
  if constexpr (kVec32) {
    ld_stream_v8(src, v[0], v[1]);
  } else {
    v[0] = ld_stream_v4(src);
    v[1] = ld_stream_v4(src + 16);
  }
}

// One lane's share of one pass: its 16 elements (two lanes per 32-element
// block) -> the block's E8M0 scale exponent.  |x| per half with
// max.xorsign.abs, sign bits cleared, then the larger half (the unsigned order
// of non-negative BF16/FP16 patterns is the order of their magnitudes), then
// the partner lane's half block.
template <bool kF16>
__device__ __forceinline__ uint32_t lane_block_scale(const uint4 (&v)[2]) {
  uint32_t h;
  if constexpr (kF16) {
    h = max_abs_f16x2(max_abs_f16x2(max_abs_f16x2(v[0].x, v[0].y), max_abs_f16x2(v[0].z, v[0].w)),
                      max_abs_f16x2(max_abs_f16x2(v[1].x, v[1].y), max_abs_f16x2(v[1].z, v[1].w)));
  } else {
    h = max_abs_bf16x2(
        max_abs_bf16x2(max_abs_bf16x2(v[0].x, v[0].y), max_abs_bf16x2(v[0].z, v[0].w)),
        max_abs_bf16x2(max_abs_bf16x2(v[1].x, v[1].y), max_abs_bf16x2(v[1].z, v[1].w)));
  }
  h &= 0x7FFF7FFFu;
  uint32_t m = max(h & 0xFFFFu, h >> 16);
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  return kF16 ? e8m0_from_absmax_f32bits(f16_bits_to_f32_bits(m)) : e8m0_from_absmax_bf16(m);
}

// The lane's 16 codes (8 bytes): x * 2^(127-s) rounded to E2M1; s == 0 gives
// zero codes.
template <bool kF16>
__device__ __forceinline__ uint2 lane_codes(const uint4 (&v)[2], uint32_t s) {
  const float inv = inv_scale_from_e8m0(s);
  uint2 code;
  if constexpr (kF16) {
    code.x = scale_cvt_e2m1x8_f16(v[0], inv);
    code.y = scale_cvt_e2m1x8_f16(v[1], inv);
  } else {
    code.x = scale_cvt_e2m1x8(v[0], inv);
    code.y = scale_cvt_e2m1x8(v[1], inv);
  }
  if (s == 0u) code = make_uint2(0u, 0u);
  return code;
}

// ------------------------------------------------ grouped segment lookup
// Segment holding padded row `prow`: the last e in [0, E) with P[e] <= prow
// (empty segments share their start with the next one, so the last such e
// is never empty when prow < P[E]).  A proportional estimate is checked
// first with two independent probes (exact whenever the segments are close to
// uniform, as with balanced MoE routing); otherwise a binary search over the
// side the estimate excluded.  P is small and read by every CTA (L1/L2 hits).
__device__ __forceinline__ int find_segment(const int32_t* __restrict__ P, int E, int prow,
                                            int total) {
  int e = static_cast<int>(static_cast<int64_t>(prow) * E / total);
  e = e < E - 1 ? e : E - 1;
  const int pe = __ldg(P + e);
  const int pn = __ldg(P + e + 1);
  if (pe <= prow && prow < pn) return e;
  int lo, hi;
  if (pe <= prow) { lo = e + 1; hi = E - 1; } else { lo = 0; hi = e - 1; }
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(P + mid) <= prow) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// L2 policy that keeps lines resident ahead of streaming traffic, and a
// 4-byte store under such a policy: for small stores that several CTAs
// complete sector by sector (a sector evicted half written costs a DRAM read
// to merge it).
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void st_keep_u32(void* p, uint32_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.u32 [%0], %1, %2;" ::"l"(p), "r"(v), "l"(pol) : "memory");
}

// L2 prefetch of the 128-byte line holding p.  It returns no data, so a
// kernel may issue it before its grid-dependency wait: the L2 is where this
// GPU's writes become coherent, so the loads after the wait read the
// predecessor's writes whatever the prefetch brought in.  Issued by the CTAs
// that start while the preceding grid drains, it fills the DRAM idle time of
// that grid's last wave.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Programmatic dependent launch: wait until the preceding grid of the stream
// has completed and its writes are visible (no-op without a predecessor),
// and allow the next grid of the stream to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace mxfp4
