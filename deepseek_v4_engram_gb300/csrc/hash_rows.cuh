// Device helpers of stages 1 and 2 shared by the kernels that hash and gather: the compressed id
// of a window position (page "Module engram", stage 1 and struct NgramHashState) and the fp8 row
// dequantisation (stage 2, embed_rows / regen_table).
#pragma once

#include "device.cuh"
#include "kernels.h"

namespace engram {

// c_{p-k} for position t of sequence b: from this call's tokens (k <= t), from the cache (earlier
// calls), or pad_id (before p = 0).
__device__ __forceinline__ int32_t compressed_id(const HashArgs& a, int32_t b, int32_t t,
                                                 int32_t len0, int32_t k) {
  if (k <= t) {
    const int32_t tok = __ldg(a.tokens + static_cast<int64_t>(b) * a.T + (t - k));
    if (tok < 0 || tok >= a.vocab) {
      set_error(a.err, kErrTokenRange);
      return a.pad_id;
    }
    return __ldg(a.token_map + tok);
  }
  const int32_t q = len0 + t - k;  // an earlier call's position
  if (q < 0) return a.pad_id;
  if (q >= a.capacity) {           // never cached (the cache was full): flagged on that call
    set_error(a.err, kErrCacheCapacity);
    return a.pad_id;
  }
  return a.cache[static_cast<int64_t>(b) * a.capacity + q];
}

// fp8 e4m3fn code -> f32, from its bit fields: sign, 4-bit exponent (bias 7), 3-bit mantissa;
// exponent 0 is subnormal (m * 2^-9); S.1111.111 is NaN. Exact.
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  const uint32_t sign = (c & 0x80u) << 24;
  const uint32_t E = (c >> 3) & 0xFu;
  const uint32_t m = c & 0x7u;
  if (E == 0xFu && m == 0x7u) return __uint_as_float(sign | 0x7FC00000u);
  if (E == 0) return __uint_as_float(sign | __float_as_uint(static_cast<float>(m) * 0x1p-9f));
  return __uint_as_float(sign | ((E + 120u) << 23) | (m << 20));
}

// e8m0 code -> 2^(code - 127) as f32 (code 0 is the binary32 subnormal 2^-127; 255 is NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t c) {
  if (c == 255u) return __uint_as_float(0x7FC00000u);
  if (c == 0u) return __uint_as_float(0x00400000u);
  return __uint_as_float(c << 23);
}

// Dequantise 16 fp8 codes (one 16-byte chunk) with one scale into 16 bf16 (two 16-byte words).
__device__ __forceinline__ void dequant16(const uint4 codes, float scale, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
  uint32_t o[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float v0 = __fmul_rn(e4m3_to_f32(w[j] & 0xFFu), scale);
    const float v1 = __fmul_rn(e4m3_to_f32((w[j] >> 8) & 0xFFu), scale);
    const float v2 = __fmul_rn(e4m3_to_f32((w[j] >> 16) & 0xFFu), scale);
    const float v3 = __fmul_rn(e4m3_to_f32(w[j] >> 24), scale);
    o[2 * j] = pack_bf16x2(v0, v1);
    o[2 * j + 1] = pack_bf16x2(v2, v3);
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

}  // namespace engram
