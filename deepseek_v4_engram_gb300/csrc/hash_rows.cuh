// Device helpers of stages 1 and 2 shared by the kernels that hash and gather: the compressed id
// of a window position (page "Module engram", stage 1 and struct NgramHashState) and the fp8 row
// dequantisation (stage 2, embed_rows / regen_table).
#pragma once

#include <cuda_fp16.h>

#include "device.cuh"
#include "kernels.h"

namespace engram {

// Read-only global loads issued exactly where they are written. A plain __ldg may be re-issued
// by the compiler at the point of use instead of keeping its result in registers (the data cannot
// change during the kernel), which puts the load's latency back on that later path; volatile asm
// is neither repeated nor moved past other volatile asm.
__device__ __forceinline__ uint4 ldg_pinned_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ldg_pinned_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg_pinned_u8(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t saddr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(saddr) : "memory");
  return v;
}

// floor((2^64 - 1) / d): the reciprocal that reduces a 64-bit value modulo d (d >= 1) with one
// high multiply (mod_u64_by).
__device__ __forceinline__ uint64_t mod_magic_u64(uint64_t d) { return d == 0 ? 0 : ~0ull / d; }

// v mod d from magic = mod_magic_u64(d) (Barrett reduction). q = floor(v * magic / 2^64) is the
// true quotient or at most 2 below it (magic >= (2^64 - 1) / d - 1 and v < 2^64), never above, so
// v - q * d lies in [0, 3d) and two conditional subtractions finish it. Exact for every v and
// every 1 <= d < 2^62.
__device__ __forceinline__ uint64_t mod_u64_by(uint64_t v, uint64_t d, uint64_t magic) {
  const uint64_t q = __umul64hi(v, magic);
  uint64_t r = v - q * d;
  if (r >= d) r -= d;
  if (r >= d) r -= d;
  return r;
}

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

// fp8 e4m3fn code -> f32, exact and branch-free. The 7 bits below the sign, placed in an IEEE
// half's exponent and mantissa fields (bits 13-7), form a half whose value is the code's magnitude
// times 2^-8 (the exponent biases are 15 and 7), for normal (E >= 1: 2^(E-7) (1 + m/8)) and
// subnormal codes (E = 0: m 2^-9) alike; S.1111.111 is NaN.
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
  const float mag =
      __half2float(__ushort_as_half(static_cast<unsigned short>((c & 0x7Fu) << 7))) * 256.0f;
  const uint32_t sign = (c & 0x80u) << 24;
  return __uint_as_float(sign | ((c & 0x7Fu) == 0x7Fu ? 0x7FC00000u : __float_as_uint(mag)));
}

// e8m0 code -> 2^(code - 127) as f32 (code 0 is the binary32 subnormal 2^-127; 255 is NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t c) {
  if (c == 255u) return __uint_as_float(0x7FC00000u);
  if (c == 0u) return __uint_as_float(0x00400000u);
  return __uint_as_float(c << 23);
}

// Dequantise 16 fp8 codes (one 16-byte chunk) with one scale into 16 bf16 (two 16-byte words).
// Each pair of codes goes to two halves with the hardware conversion (exact: every e4m3 value,
// subnormals included, is a half), then to f32, times the e8m0 scale (a power of two: exact
// unless the product leaves the f32 range), rounded to bf16 (exact for the same reason: 4
// significant bits).
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
