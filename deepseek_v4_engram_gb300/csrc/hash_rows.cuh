// Device helpers of stages 1 and 2 shared by the kernels that hash and gather: the compressed id
// of a window position (page "Module engram", stage 1 and struct NgramHashState) and the fp8 row
// dequantisation (stage 2, embed_rows / regen_table).
#pragma once

#include <cuda_fp16.h>

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

// Read-only loads of table rows and scales with an L2 cache policy: a gathered row is read once,
// so it is marked evict-first and later misses replace it rather than lines other kernels left
// (measured 3% faster for the four-layer gather at 4096 tokens, 0.4% for the prefill step).
__device__ __forceinline__ uint4 ldg_hint(const uint4* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}
__device__ __forceinline__ uint32_t ldg_u8_hint(const uint8_t* p, uint64_t policy) {
  uint16_t v;
  asm volatile("ld.global.nc.L2::cache_hint.u8 %0, [%1], %2;" : "=h"(v) : "l"(p), "l"(policy));
  return v;
}

// e8m0 code -> 2^(code - 127) as f32 (code 0 is the binary32 subnormal 2^-127; 255 is NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t c) {
  if (c == 255u) return __uint_as_float(0x7FC00000u);
  if (c == 0u) return __uint_as_float(0x00400000u);
  return __uint_as_float(c << 23);
}

// Dequantise 16 fp8 e4m3fn codes (one 16-byte chunk) with one scale into 16 bf16 (two 16-byte
// words). Each pair of codes goes to two halves with the hardware conversion (exact: every e4m3
// value, subnormals included, is a half; S.1111.111 becomes NaN), then to f32, times the e8m0
// scale (a power of two: exact unless the product leaves the f32 range), rounded to bf16 (exact
// for the same reason: 4 significant bits).
__device__ __forceinline__ void dequant16(const uint4 codes, float scale, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
  uint32_t o[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const uint16_t pair = static_cast<uint16_t>(w[j] >> (16 * half));
      uint32_t h2;
      asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
      o[2 * j + half] = pack_bf16x2(__fmul_rn(f.x, scale), __fmul_rn(f.y, scale));
    }
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

}  // namespace engram
