// Launch interface of the decode step (decode_step_sm103.cu) and its gate kernel (stages.cu).
// Host-only declarations; every pointer is a device pointer already validated by capi.cu.
#pragma once

#include "kernels.h"

namespace engram {

// The decode step's stages 1-3 in one kernel (decode_step_sm103.cu): hash + gather inside every
// CTA, the weight streamed over every SM, key partial sums and value rows out.
struct DecodeStepArgs {
  HashArgs hash;          // tokens, cache, tables, optional hash_ids out (unused when ids given)
  const int32_t* ids;     // [M, S] given hash ids, or null to hash the tokens
  const uint8_t* table;   // [num_rows, 64] e4m3
  const uint8_t* scales;  // [num_rows, 2] e8m0 (2-byte aligned)
  int64_t num_rows;
  const uint16_t* w;      // [N, K]
  const uint16_t* x;      // [M, hc, dim]
  const uint16_t* q;      // [hc, dim]
  const uint16_t* k;      // [hc, dim]
  float2* part;           // [hc * dim / 32, 64]: per 32-column key group and token, (sum key^2,
                          // sum h * w * key)
  uint16_t* value;        // [M, dim] bf16
  uint16_t* kv_out;       // [M, N] or null
  int64_t M;
  int32_t N, K, hc, dim;
  int32_t nt;             // tokens rounded up to 32 (set by launch_decode_step)
  uint32_t* err;
};

struct DecodeGeometry {
  int32_t dim, hc, n_heads, max_ngram, head_dim;
};

// Stage 4 from the decode step's partial sums: one block per (token, stream).
struct GatePartArgs {
  const uint16_t* x;      // [M, hc, dim]
  const float2* part;     // as DecodeStepArgs::part
  const uint16_t* value;  // [M, dim]
  const uint8_t* mask;    // [M] or null
  uint16_t* out;          // [M, hc, dim]
  float* gate_out;        // [M, hc] or null
  int64_t M;
  int32_t hc, dim;
  float eps;
  float inv_sqrt_dim;
  LenAdvance adv;         // adv.len may be null
};

// The decode step (M <= 64, head_dim 64): decode_step_part_bytes of partial sums and M * dim
// bf16 value rows of scratch.
bool decode_step_supported(int64_t M, const DecodeGeometry& g);
size_t decode_step_part_bytes(int32_t hc, int32_t dim);
cudaError_t launch_decode_step(const DecodeStepArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_gate_part(const GatePartArgs& a, cudaStream_t s, bool pdl = false);

}  // namespace engram
