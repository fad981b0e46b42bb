// Internal launch interface between the C ABI (capi.cu) and the kernel translation units.
// Host-only declarations; every pointer is a device pointer already validated by capi.cu.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include <utility>

#include "engram.h"

namespace engram {

struct HashArgs {
  const int32_t* tokens;     // [B, T]
  int32_t B, T;
  int32_t* cache;            // [B, capacity]
  const int32_t* cache_len;  // [B], read only here
  int32_t capacity;
  int32_t* hash_ids;         // [B, T, S]
  const int32_t* token_map;
  int32_t vocab, pad_id;
  const uint64_t* multipliers;  // [max_ngram]
  const uint64_t* primes;       // [S]
  const int64_t* offsets;       // [S]
  int32_t n_heads, max_ngram;
  uint32_t* err;
};

// One Engram layer's share of the hash + gather kernel: its own hash constants and table.
struct HashLayer {
  const uint64_t* multipliers;  // [max_ngram]
  const uint64_t* primes;       // [S]
  const int64_t* offsets;       // [S]
  const uint8_t* table;         // [num_rows, hd] e4m3
  const uint8_t* scales;        // [num_rows, hd/32] e8m0
  int64_t num_rows;
  uint16_t* rows;               // [B*T, S, hd] bf16
  int32_t* hash_ids;            // [B*T, S] or null (ids then stay in registers)
};

constexpr int kMaxHashLayers = ENGRAM_MAX_HASH_LAYERS;

// Stages 1 + 2 in one kernel for n_layers layers: the window of each position (token map, cache,
// pad) is resolved once, then every layer hashes it with its own constants and gathers +
// dequantises its own rows. hash.multipliers / primes / offsets / hash_ids are not read (each
// layer's are in `layer`).
struct HashRowsArgs {
  HashArgs hash;
  int32_t n_layers;
  int32_t head_dim;
  HashLayer layer[kMaxHashLayers];
  int32_t* zero;          // optional: zero_n int32 set to 0 (the next kernel's counters)
  int32_t zero_n;
  int32_t positions;      // positions per block (set by launch_hash_rows)
};

// The single-layer form: layer 0 takes the constants and ids of `h` and the given table.
HashRowsArgs single_layer_hash_rows(const HashArgs& h, const uint8_t* table,
                                    const uint8_t* scales, int64_t num_rows, int32_t head_dim,
                                    uint16_t* rows);

// Advance cache_len[b] += T (clamped to capacity) for b < B; done by one block of the last kernel
// of the forward, once every reader of the old lengths has finished.
struct LenAdvance {
  int32_t* len;
  int32_t B, T, cap;
};

struct RowsArgs {
  const uint8_t* table;   // [rows, hd] e4m3
  const uint8_t* scales;  // [rows, hd/32] e8m0
  const int32_t* ids;     // [n_ids]
  int64_t n_ids;
  int64_t num_rows;
  int32_t head_dim;
  uint16_t* out;          // [n_ids, hd] bf16
  // Optional: advance cache_len[b] += T for b < adv_B (done by block 0), used by the forward to
  // fold the cache-length update into a kernel that runs after the hash.
  int32_t* adv_len;
  int32_t adv_B, adv_T, adv_cap;
  uint32_t* err;
  int32_t* zero;          // optional: zero_n int32 set to 0 (the next kernel's counters)
  int32_t zero_n;
};

struct GateArgs {
  const uint16_t* x;    // [M, hc, dim]
  const uint16_t* kv;   // [M, dim*(hc+1)] bf16, or null when `part` is given
  const float* part;    // [ksplit, M, dim*(hc+1)] f32 partial sums of kv, or null
  int32_t ksplit;
  uint16_t* kv_out;     // [M, dim*(hc+1)] or null: kv as used (bf16)
  const uint16_t* q;    // [hc, dim]
  const uint16_t* k;    // [hc, dim]
  const uint8_t* mask;  // [M] or null
  uint16_t* out;        // [M, hc, dim]
  float* gate_out;      // [M, hc] or null
  int64_t M;
  int32_t hc, dim;
  float eps;
  float inv_sqrt_dim;
  LenAdvance adv;       // adv.len may be null
};

struct WkvArgs {
  const uint16_t* a;  // [M, K]
  const uint16_t* w;  // [N, K]
  uint16_t* kv;       // [M, N]
  int64_t M;
  int32_t N, K;
  uint32_t* err;
};

struct WkvSmallArgs {
  const uint16_t* a;  // [M, K] (M <= 256)
  const uint16_t* w;  // [N, K]
  uint16_t* kv;       // [M, N] bf16 when ksplit == 1
  float* part;        // [ksplit, M, N] f32 when ksplit > 1
  int64_t M;
  int32_t N, K, ksplit;
  uint32_t* err;
};

struct FusedArgs {
  const uint16_t* a;      // [M, K] gathered rows (bf16)
  const uint16_t* w;      // [N, K]
  const uint16_t* x;      // [M, hc, dim]
  const uint16_t* q;      // [hc, dim]
  const uint16_t* k;      // [hc, dim]
  const uint8_t* mask;    // [M] or null
  uint16_t* out;          // [M, hc, dim]
  float* gate_out;        // [M, hc] or null
  uint16_t* kv_out;       // [M, N] or null
  int64_t M;
  int32_t K, hc, dim;
  float eps, inv_sqrt_dim;
  uint32_t* err;
  LenAdvance adv;         // adv.len may be null
  void* scratch;          // fused_scratch_bytes(M, hc, dim) bytes, 256-byte aligned
  bool sync_cleared;      // the scratch's counters were cleared by the previous kernel
  uint16_t* vout;         // [M, dim] or null. Set: deferred output: value tiles store their bf16
                          // value rows here and do not write out (launch_gate_apply does, after)
};

// out = h + gate * value from the gates and value rows the fused kernel left in its deferred
// output mode: one block per (token, stream).
struct GateApplyArgs {
  const uint16_t* x;      // [M, hc, dim]
  const float* gx;        // [M, hc] gates (0 for a masked token)
  const uint16_t* value;  // [M, dim] bf16
  const uint8_t* mask;    // [M] or null
  uint16_t* out;          // [M, hc, dim]
  int64_t M;
  int32_t hc, dim;
};

// The counters in the fused kernel's scratch that must be zero when it starts.
void fused_sync_region(void* scratch, int64_t M, int32_t hc, int32_t dim, int32_t** ptr,
                       int32_t* count);

// `pdl`: launch with programmatic stream serialization (the kernel then overlaps its launch and
// prologue with the previous kernel of the stream and waits for it before touching its data).
cudaError_t launch_hash_rows(const HashRowsArgs& a, cudaStream_t s, bool pdl);
cudaError_t launch_hash(const HashArgs& a, cudaStream_t s);
cudaError_t launch_advance_len(int32_t* cache_len, int32_t B, int32_t T, int32_t cap,
                               cudaStream_t s);
cudaError_t launch_rows(const RowsArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_gate(const GateArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_wkv(const WkvArgs& a, cudaStream_t s, bool pdl = false);
bool small_supported(int64_t M, int32_t N, int32_t K);
int small_ksplit(int32_t N, int32_t K);
cudaError_t launch_wkv_small(const WkvSmallArgs& a, cudaStream_t s, bool pdl = false);
// Weight-streaming projection for M <= 64 tokens (decode): bf16 kv, no partial sums.
bool decode_supported(int64_t M, int32_t N, int32_t K);
cudaError_t launch_wkv_decode(const WkvSmallArgs& a, cudaStream_t s, bool pdl = false);
bool fused_supported(int32_t K, int32_t hc, int32_t dim);
size_t fused_scratch_bytes(int64_t M, int32_t hc, int32_t dim);
// The gates [M, hc] f32 at the start of the fused kernel's scratch.
const float* fused_gates(const void* scratch);
cudaError_t launch_gate_apply(const GateApplyArgs& a, cudaStream_t s, bool pdl = false);
cudaError_t launch_fused(const FusedArgs& a, cudaStream_t s, bool pdl = false);

// cudaLaunchKernelEx with optional programmatic stream serialization.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t st, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Host-side state per device (capi.cu), thread-safe: the current device's SM count, and raising
// a kernel's dynamic shared-memory limit once per (device, kernel) (the limit is a property of
// the function on each device, so a process that drives several GPUs needs it on every one).
int device_sm_count();
cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes);

// The fused kernel's resident CTA pairs on the current device (forward_sm103.cu), cached per
// device.
int fused_resident_pairs_cached(int (*query)());

// Smallest workspace engram_forward accepts for M tokens (the fused path's, where it applies).
size_t forward_min_workspace_bytes(const engram_desc_t* desc, int64_t M);

// Sets the message engram_last_error() returns on this thread; returns `code`.
int set_last_error(int code, const char* msg);

// Tensor maps (capi.cu; cuTensorMapEncodeTiled is fetched from the driver on first use).
bool tensor_map_2d_bf16(void* map_out, const void* base, uint64_t inner, uint64_t rows,
                        uint32_t box_inner, uint32_t box_rows);
// 3-D bf16 tensor [d2][d1][d0] (d0 innermost, dense), 128-byte swizzle.
bool tensor_map_3d_bf16(void* map_out, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                        uint32_t box0, uint32_t box1, uint32_t box2);

}  // namespace engram
