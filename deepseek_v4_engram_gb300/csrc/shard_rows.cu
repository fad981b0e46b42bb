// Stage 2 (page "Module engram", stage 2 / embed_rows) on one rank's share of a row-sharded table.
//
// A row this rank holds is gathered and dequantised as by engram_embed_rows. A row another rank
// holds is written as bf16 -0.0 in every element: -0 is the identity of IEEE addition
// (-0 + v = v for every v, +0 and -0 included), so the sum over ranks of their outputs, in any
// order, is the unsharded gather bit for bit. (A +0 fill would turn the -0 that e4m3 code 0x80
// dequantises to into +0.)
#include "device.cuh"
#include "hash_rows.cuh"
#include "shard.h"

namespace engram {

__global__ void __launch_bounds__(256) shard_rows_kernel(ShardRowsArgs a) {
  const int32_t chunks = a.head_dim / 16;
  const int64_t total = a.n_ids * chunks;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / chunks;
    const int32_t c = static_cast<int32_t>(i % chunks);
    const int32_t id = __ldg(a.ids + r);
    const int64_t local = static_cast<int64_t>(id) - a.row_begin;
    uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
    if (local >= 0 && local < a.shard_rows) {
      const uint4 codes = __ldg(reinterpret_cast<const uint4*>(a.table + local * a.head_dim +
                                                               c * 16));
      const uint32_t sc = __ldg(a.scales + local * (a.head_dim / 32) + c / 2);
      dequant16(codes, e8m0_to_f32(sc), lo, hi);
    } else if (id >= 0 && id < a.num_rows) {
      lo = make_uint4(0x80008000u, 0x80008000u, 0x80008000u, 0x80008000u);   // another rank's row
      hi = lo;
    } else {
      set_error(a.err, kErrIdRange);   // a zero row, as the unsharded gather writes
    }
    uint4* dst = reinterpret_cast<uint4*>(a.out + r * a.head_dim + c * 16);
    dst[0] = lo;
    dst[1] = hi;
  }
}

cudaError_t launch_shard_rows(const ShardRowsArgs& a, cudaStream_t st) {
  const int64_t total = a.n_ids * (a.head_dim / 16);
  int64_t blocks = (total + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > (1 << 20)) blocks = 1 << 20;   // grid-stride beyond
  shard_rows_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace engram
