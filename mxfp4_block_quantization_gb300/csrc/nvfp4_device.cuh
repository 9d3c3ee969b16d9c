// nvfp4_device.cuh — the NVFP4 block steps shared by the dense, grouped and
// dispatch-fused NVFP4 kernels (nvfp4.cu, dispatch.cu).
//
// Method: vLLM PR #43557 page, "Implementation breakdown" item 1 (the
// non-UE8M0 branch of cvt_warp_fp16_to_fp4) and "Review highlights" (the
// elements are scaled with the E4M3-rounded scale).  Every step one float32
// operation rounded to nearest even: q = vecMax / 6; byte = E4M3(g * q);
// inv = g / float(byte); code = E2M1(x * inv); byte 0 -> zero codes.
#pragma once

#include <cstdint>

#include "mxfp4_device.cuh"

namespace mxfp4 {

// The block's 8 code bytes: x * inv rounded to E2M1, inv = g / float(byte);
// zero codes for byte 0.
template <bool kF16>
__device__ __forceinline__ uint2 nv_codes(const uint4 (&v)[2], uint32_t byte, float inv) {
  uint2 code = make_uint2(0u, 0u);
  if (byte != 0u) {
    if constexpr (kF16) {
      code.x = scale_cvt_e2m1x8_f16(v[0], inv);
      code.y = scale_cvt_e2m1x8_f16(v[1], inv);
    } else {
      code.x = scale_cvt_e2m1x8(v[0], inv);
      code.y = scale_cvt_e2m1x8(v[1], inv);
    }
  }
  return code;
}

// The block's q = vecMax / 6 (the part of the scale that does not depend on
// the global scale).
template <bool kF16>
__device__ __forceinline__ float nv_block_q(const uint4 (&v)[2]) {
  uint32_t h;
  if constexpr (kF16) {
    h = max_abs_f16x2(max_abs_f16x2(max_abs_f16x2(v[0].x, v[0].y), max_abs_f16x2(v[0].z, v[0].w)),
                      max_abs_f16x2(max_abs_f16x2(v[1].x, v[1].y), max_abs_f16x2(v[1].z, v[1].w)));
  } else {
    h = max_abs_bf16x2(max_abs_bf16x2(max_abs_bf16x2(v[0].x, v[0].y),
                                      max_abs_bf16x2(v[0].z, v[0].w)),
                       max_abs_bf16x2(max_abs_bf16x2(v[1].x, v[1].y),
                                      max_abs_bf16x2(v[1].z, v[1].w)));
  }
  h &= 0x7FFF7FFFu;
  const uint32_t m = max(h & 0xFFFFu, h >> 16);
  return __uint_as_float(kF16 ? f16_bits_to_f32_bits(m) : m << 16) / 6.0f;  // IEEE division
}

// One lane's 16-element block -> its E4M3 scale byte: byte = E4M3(g * q).
template <bool kF16>
__device__ __forceinline__ uint32_t nv_scale_byte(const uint4 (&v)[2], float g) {
  return cvt_e4m3_satfinite(g * nv_block_q<kF16>(v));
}

}  // namespace mxfp4
