// Stage 2 over a row-sharded table (Engram listing, __init__: the embedding is a
// ParallelEngramEmbedding): each rank holds a contiguous range of the table's rows.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace engram {

struct ShardRowsArgs {
  const uint8_t* table;    // [shard_rows, hd] e4m3: rows row_begin .. row_begin + shard_rows - 1
  const uint8_t* scales;   // [shard_rows, hd/32] e8m0
  const int32_t* ids;      // [n_ids] global row ids
  int64_t n_ids;
  int64_t row_begin;
  int64_t shard_rows;
  int64_t num_rows;        // rows of the whole table
  int32_t head_dim;
  uint16_t* out;           // [n_ids, hd] bf16
  uint32_t* err;
};

cudaError_t launch_shard_rows(const ShardRowsArgs& a, cudaStream_t st);

}  // namespace engram
