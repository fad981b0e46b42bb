// C ABI of the Engram forward path: argument validation, the device error word, tensor maps, and
// the launch sequence of each entry point. Declared in include/engram.h.
#include <cstdarg>
#include <cstdio>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "engram.h"
#include "kernels.h"
#include "shard.h"
#include "stream_probe.h"

namespace engram {

// One error word per device (each device that loads the library has its own copy).
__device__ uint32_t g_error_word;

namespace {

thread_local char g_msg[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(ENGRAM_ECUDA, "%s: %s", where, cudaGetErrorString(e));
}

int cuda_fail(cudaError_t e, const char* who, const char* stage) {
  return fail(ENGRAM_ECUDA, "%s: %s: %s", who, stage, cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;

// Per-device host state (device_sm_count, ensure_dynamic_smem, fused_resident_pairs_cached).
std::mutex g_dev_mu;
int g_sm_count[kMaxDevices] = {};
int g_fused_pairs[kMaxDevices] = {};
constexpr int kMaxSmemKernels = 16;
const void* g_smem_kernel[kMaxDevices][kMaxSmemKernels] = {};

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = 0;
  return dev;
}
uint32_t* g_err_ptr[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Device address of this device's error word (resolved once per device, with it current).
uint32_t* error_word(cudaError_t* e_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *e_out = e != cudaSuccess ? e : cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_err_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_error_word);
    if (e != cudaSuccess) {
      *e_out = e;
      return nullptr;
    }
    g_err_ptr[dev] = static_cast<uint32_t*>(p);
  }
  *e_out = cudaSuccess;
  return g_err_ptr[dev];
}

bool aligned(const void* p, size_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

int check_desc(const engram_desc_t* d) {
  if (d == nullptr) return fail(ENGRAM_EINVAL, "desc is NULL");
  if (d->dim <= 0 || d->hc_mult <= 0 || d->n_heads <= 0 || d->head_dim <= 0)
    return fail(ENGRAM_EINVAL, "dim, hc_mult, n_heads and head_dim must be > 0");
  if (d->max_ngram_size < 2 || d->max_ngram_size > 8)
    return fail(ENGRAM_EINVAL, "max_ngram_size must be in [2, 8]");
  if (d->head_dim % 32 != 0)
    return fail(ENGRAM_EINVAL, "head_dim must be a multiple of 32 (one e8m0 scale per 32)");
  if (d->dim % 8 != 0) return fail(ENGRAM_EINVAL, "dim must be a multiple of 8");
  if (d->num_embeddings <= 0 || d->num_embeddings >= (int64_t(1) << 31))
    return fail(ENGRAM_EINVAL, "num_embeddings must be in [1, 2^31)");
  if (!(d->norm_eps >= 0.0f)) return fail(ENGRAM_EINVAL, "norm_eps must be >= 0");
  const int64_t S = int64_t(d->max_ngram_size - 1) * d->n_heads;
  if (S * d->head_dim >= (int64_t(1) << 30) || int64_t(d->dim) * (d->hc_mult + 1) >= (1 << 30))
    return fail(ENGRAM_EINVAL, "projection too large");
  return ENGRAM_OK;
}

int check_tables(const engram_tables_t* t) {
  if (t == nullptr) return fail(ENGRAM_EINVAL, "tables is NULL");
  if (!t->token_map || !t->multipliers || !t->primes || !t->offsets)
    return fail(ENGRAM_EINVAL, "a table pointer is NULL");
  if (t->vocab <= 0 || t->pad_id < 0) return fail(ENGRAM_EINVAL, "vocab must be > 0, pad_id >= 0");
  if (!aligned(t->token_map, 4) || !aligned(t->multipliers, 8) || !aligned(t->primes, 8) ||
      !aligned(t->offsets, 8))
    return fail(ENGRAM_EINVAL, "misaligned table pointer");
  return ENGRAM_OK;
}

int n_hash_cols(const engram_desc_t* d) { return (d->max_ngram_size - 1) * d->n_heads; }

// ids may be NULL only when ids_optional (the forward then hashes into its workspace).
int hash_checks(const engram_desc_t* d, const engram_tables_t* t, const int32_t* tokens,
                int32_t B, int32_t T, int32_t* cache, int32_t* cache_len, int32_t cap,
                int32_t* ids, bool ids_optional = false) {
  int rc = check_desc(d);
  if (rc) return rc;
  rc = check_tables(t);
  if (rc) return rc;
  if (B < 0 || T < 0 || cap < 0) return fail(ENGRAM_EINVAL, "B, T and capacity must be >= 0");
  if (int64_t(B) * T * n_hash_cols(d) >= (int64_t(1) << 39))
    return fail(ENGRAM_EINVAL, "B * T too large");
  if (B * int64_t(T) == 0) return ENGRAM_OK;
  if (!tokens || !cache || !cache_len || (!ids && !ids_optional))
    return fail(ENGRAM_EINVAL, "NULL array");
  if (!aligned(tokens, 4) || !aligned(cache, 4) || !aligned(cache_len, 4) || !aligned(ids, 4))
    return fail(ENGRAM_EINVAL, "misaligned int32 array");
  if (ids && overlaps(ids, size_t(B) * T * n_hash_cols(d) * 4, cache, size_t(B) * cap * 4))
    return fail(ENGRAM_EINVAL, "hash_ids overlaps cache");
  return ENGRAM_OK;
}

HashArgs make_hash_args(const engram_desc_t* d, const engram_tables_t* t, const int32_t* tokens,
                        int32_t B, int32_t T, int32_t* cache, int32_t* cache_len, int32_t cap,
                        int32_t* ids, uint32_t* err) {
  HashArgs h{};
  h.tokens = tokens;
  h.B = B;
  h.T = T;
  h.cache = cache;
  h.cache_len = cache_len;
  h.capacity = cap;
  h.hash_ids = ids;
  h.token_map = t->token_map;
  h.vocab = t->vocab;
  h.pad_id = t->pad_id;
  h.multipliers = t->multipliers;
  h.primes = t->primes;
  h.offsets = t->offsets;
  h.n_heads = d->n_heads;
  h.max_ngram = d->max_ngram_size;
  h.err = err;
  return h;
}

constexpr size_t round256(size_t n) { return (n + 255) & ~size_t(255); }

// How engram_forward runs stages 3 and 4 for a given token count, fastest first:
//  - kDecode:  M <= 64: weight-streaming projection in 64-row units, a fixed share per SM, into
//              a bf16 kv (no partial sums), then the gate kernel;
//  - kSmall:   M <= 256: weight-streaming projection over every SM (split-K partials in f32 when
//              the workspace holds them, else bf16 kv), then the gate kernel;
//  - kUnfused: the persistent projection GEMM into a bf16 kv, then the gate kernel; measured
//              faster than the fused kernel below 640 tokens (too few items to fill the GPU
//              past the fused kernel's cold start: 72 vs 74 us at 512, 86 vs 82 us at 640);
//  - kFusedDeferred: 240-256 and 512-2048 tokens: the fused kernel with deferred output: its value
//              tiles store bf16 value rows instead of waiting for the gates, and a light kernel
//              then writes out = x + gate * value; for batches too small for the fused kernel to
//              hide its value tiles' wait and x traffic behind the key tiles of other token
//              tiles;
//  - kFused:   projection + gate in one kernel; kv never touches HBM; least workspace.
enum class Path { kDecode, kSmall, kUnfused, kFusedDeferred, kFused };
struct Plan {
  Path path;
  int ksplit;
  size_t bytes;
};
constexpr int64_t kFusedMinTokens = 640;
// Where the deferred-output fused plan is the fastest, measured on one GPU against the other
// plans (whole engram_forward, B1): one nearly full token tile, 51.2-51.8 vs 54.0-54.1 us at 256
// tokens (54.0 vs 53.9 at 240: the small-batch plan grows with M, the fused kernel's one tile
// does not); and 512 to 2048 tokens, 63.2 vs 70.0 at 512, 96.1 vs 105.3 at 1024, 145.7 vs 157.6
// at 2048. Slower at 288-384 (61.4 vs 54.0 at 288: a second, nearly empty tile) and from 3072
// (213.7 vs 205.9; 272.7 vs 266.3 at 4096).
bool deferred_plan_wins(int64_t M) { return (M >= 240 && M <= 256) || (M >= 512 && M <= 2048); }
constexpr int kMaxPlans = 6;

// Candidate plans in order of preference; returns how many were written.
int forward_plans(const engram_desc_t* d, int64_t M, Plan* out) {
  const size_t S = n_hash_cols(d);
  const int32_t K = static_cast<int32_t>(S) * d->head_dim;
  const int32_t N = d->dim * (d->hc_mult + 1);
  const size_t base = round256(size_t(M) * K * 2);   // gathered rows (hash ids stay on chip)
  const size_t kv_bytes = round256(size_t(M) * N * 2);
  const bool fused = fused_supported(K, d->hc_mult, d->dim);
  int n = 0;
  if (decode_supported(M, N, K)) out[n++] = {Path::kDecode, 1, base + kv_bytes};
  if (fused && deferred_plan_wins(M))
    out[n++] = {Path::kFusedDeferred, 1,
                base + round256(fused_scratch_bytes(M, d->hc_mult, d->dim)) +
                    round256(size_t(M) * d->dim * 2)};
  if (small_supported(M, N, K)) {
    // split-K only while its f32 partial sums stay small (decode-sized batches)
    const int ks = M <= 64 ? small_ksplit(N, K) : 1;
    if (ks > 1) out[n++] = {Path::kSmall, ks, base + round256(size_t(ks) * M * N * 4)};
    out[n++] = {Path::kSmall, 1, base + kv_bytes};
  }
  if (!fused || M < kFusedMinTokens) out[n++] = {Path::kUnfused, 1, base + kv_bytes};
  if (fused) out[n++] = {Path::kFused, 1, base + fused_scratch_bytes(M, d->hc_mult, d->dim)};
  if (fused && M >= kFusedMinTokens) out[n++] = {Path::kUnfused, 1, base + kv_bytes};
  return n;
}

}  // namespace

namespace {
bool have_encoder() {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return true;
}
}  // namespace

int device_sm_count() {
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes) {
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(g_dev_mu);
  int free_slot = -1;
  for (int i = 0; i < kMaxSmemKernels; ++i) {
    if (g_smem_kernel[dev][i] == kernel) return cudaSuccess;
    if (g_smem_kernel[dev][i] == nullptr && free_slot < 0) free_slot = i;
  }
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(bytes));
  if (e == cudaSuccess && free_slot >= 0) g_smem_kernel[dev][free_slot] = kernel;
  return e;
}

int fused_resident_pairs_cached(int (*query)()) {
  const int dev = current_device();
  {
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (g_fused_pairs[dev] > 0) return g_fused_pairs[dev];
  }
  const int n = query();   // needs the kernel's shared-memory limit raised (its own lock)
  std::lock_guard<std::mutex> lock(g_dev_mu);
  g_fused_pairs[dev] = n;
  return n;
}

bool tensor_map_3d_bf16(void* map_out, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                        uint32_t box0, uint32_t box1, uint32_t box2) {
  if (!have_encoder()) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const cuuint32_t box[3] = {box0, box1, box2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(static_cast<CUtensorMap*>(map_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              3, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool tensor_map_2d_bf16(void* map_out, const void* base, uint64_t inner, uint64_t rows,
                        uint32_t box_inner, uint32_t box_rows) {
  if (!have_encoder()) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(static_cast<CUtensorMap*>(map_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Smallest workspace engram_forward accepts for M tokens (0 for an invalid descriptor).
size_t forward_min_workspace_bytes(const engram_desc_t* desc, int64_t M) {
  if (check_desc(desc) != ENGRAM_OK || M < 0) return 0;
  Plan plans[kMaxPlans];
  const int n = forward_plans(desc, M, plans);
  size_t best = 0;
  for (int i = 0; i < n; ++i)
    if (i == 0 || plans[i].bytes < best) best = plans[i].bytes;
  return best;
}

// Record a failure message for engram_last_error() from another translation unit.
int set_last_error(int code, const char* msg) { return fail(code, "%s", msg); }

}  // namespace engram

using namespace engram;

extern "C" {

ENGRAM_API const char* engram_last_error(void) { return g_msg; }

ENGRAM_API int32_t engram_abi_version(void) { return ENGRAM_ABI_VERSION; }

ENGRAM_API int engram_check_errors(void* stream, uint32_t* bits_out) {
  g_msg[0] = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "engram_check_errors: stream");
  uint32_t* w = error_word(&e);
  if (!w) return cuda_fail(e, "engram_check_errors: error word");
  uint32_t bits = 0;
  if ((e = cudaMemcpyAsync(&bits, w, 4, cudaMemcpyDeviceToHost, st)) != cudaSuccess ||
      (e = cudaMemsetAsync(w, 0, 4, st)) != cudaSuccess ||
      (e = cudaStreamSynchronize(st)) != cudaSuccess)
    return cuda_fail(e, "engram_check_errors: read");
  if (bits_out) *bits_out = bits;
  if (bits == 0) return ENGRAM_OK;
  if (bits == ENGRAM_DEVERR_CACHE_FULL)
    return fail(ENGRAM_ECAPACITY, "a look-back cache ran out of capacity");
  return fail(ENGRAM_EDEVICE, "device error word 0x%x (1 token range, 2 cache full, 4 id range, "
              "8 wait timeout)", bits);
}

ENGRAM_API int engram_hash(const engram_desc_t* desc, const engram_tables_t* tables,
                           const int32_t* tokens, int32_t B, int32_t T, int32_t* cache,
                           int32_t* cache_len, int32_t capacity, int32_t* hash_ids,
                           void* stream) {
  g_msg[0] = 0;
  int rc = hash_checks(desc, tables, tokens, B, T, cache, cache_len, capacity, hash_ids);
  if (rc) return rc;
  if (int64_t(B) * T == 0) return ENGRAM_OK;
  cudaError_t e;
  uint32_t* err = error_word(&e);
  if (!err) return cuda_fail(e, "engram_hash");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const HashArgs h = make_hash_args(desc, tables, tokens, B, T, cache, cache_len, capacity,
                                    hash_ids, err);
  if ((e = launch_hash(h, st)) != cudaSuccess) return cuda_fail(e, "engram_hash: hash kernel");
  if ((e = launch_advance_len(cache_len, B, T, capacity, st)) != cudaSuccess)
    return cuda_fail(e, "engram_hash: length update");
  return ENGRAM_OK;
}

ENGRAM_API int engram_hash_rows_layers(const engram_desc_t* desc, const engram_tables_t* tables,
                                       const engram_layer_hash_t* layers, int32_t n_layers,
                                       const int32_t* tokens, int32_t B, int32_t T,
                                       int32_t* cache, int32_t* cache_len, int32_t capacity,
                                       void* stream) {
  g_msg[0] = 0;
  if (desc == nullptr || tables == nullptr) return fail(ENGRAM_EINVAL, "desc or tables is NULL");
  if (layers == nullptr || n_layers < 1 || n_layers > ENGRAM_MAX_HASH_LAYERS)
    return fail(ENGRAM_EINVAL, "layers must hold 1 to %d layer records", ENGRAM_MAX_HASH_LAYERS);
  for (int32_t l = 0; l < n_layers; ++l) {
    const engram_layer_hash_t& L = layers[l];
    if (!L.multipliers || !L.primes || !L.offsets || !L.table || !L.scales)
      return fail(ENGRAM_EINVAL, "layer %d: a NULL pointer", l);
    if (!aligned(L.multipliers, 8) || !aligned(L.primes, 8) || !aligned(L.offsets, 8) ||
        !aligned(L.table, 16) || !aligned(L.rows, 16) || !aligned(L.hash_ids, 4))
      return fail(ENGRAM_EINVAL, "layer %d: a misaligned pointer", l);
    if (L.num_embeddings <= 0 || L.num_embeddings >= (int64_t(1) << 31))
      return fail(ENGRAM_EINVAL, "layer %d: num_embeddings must be in [1, 2^31)", l);
  }
  // the checks of engram_hash, with layer 0's constants standing in for the tables' own
  engram_desc_t d = *desc;
  d.num_embeddings = layers[0].num_embeddings;
  engram_tables_t t = *tables;
  t.multipliers = layers[0].multipliers;
  t.primes = layers[0].primes;
  t.offsets = layers[0].offsets;
  int rc = hash_checks(&d, &t, tokens, B, T, cache, cache_len, capacity, nullptr,
                       /*ids_optional=*/true);
  if (rc) return rc;
  const int64_t M = int64_t(B) * T;
  if (M == 0) return ENGRAM_OK;
  if (M >= (int64_t(1) << 31)) return fail(ENGRAM_EINVAL, "B * T too large");
  const int S = n_hash_cols(&d);
  const size_t cache_bytes = size_t(B) * capacity * 4;
  for (int32_t l = 0; l < n_layers; ++l) {
    const engram_layer_hash_t& L = layers[l];
    if (L.rows == nullptr) return fail(ENGRAM_EINVAL, "layer %d: rows is NULL", l);
    const size_t row_bytes = size_t(M) * S * d.head_dim * 2, id_bytes = size_t(M) * S * 4;
    if (overlaps(L.rows, row_bytes, cache, cache_bytes) ||
        overlaps(L.rows, row_bytes, cache_len, size_t(B) * 4) ||
        (L.hash_ids && (overlaps(L.hash_ids, id_bytes, cache, cache_bytes) ||
                        overlaps(L.hash_ids, id_bytes, cache_len, size_t(B) * 4))))
      return fail(ENGRAM_EINVAL, "layer %d: an output overlaps the cache", l);
  }
  cudaError_t e;
  uint32_t* err = error_word(&e);
  if (!err) return cuda_fail(e, "engram_hash_rows_layers");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  HashRowsArgs a{};
  a.hash = make_hash_args(&d, &t, tokens, B, T, cache, cache_len, capacity, nullptr, err);
  a.n_layers = n_layers;
  a.head_dim = d.head_dim;
  for (int32_t l = 0; l < n_layers; ++l) {
    const engram_layer_hash_t& L = layers[l];
    a.layer[l] = HashLayer{L.multipliers, L.primes,         L.offsets, L.table,
                           L.scales,      L.num_embeddings, L.rows,    L.hash_ids};
  }
  if ((e = launch_hash_rows(a, st, true)) != cudaSuccess)
    return cuda_fail(e, "engram_hash_rows_layers: hash + rows");
  if ((e = launch_advance_len(cache_len, B, T, capacity, st)) != cudaSuccess)
    return cuda_fail(e, "engram_hash_rows_layers: length update");
  return ENGRAM_OK;
}

ENGRAM_API int engram_embed_rows(const engram_desc_t* desc, const uint8_t* table,
                                 const uint8_t* scales, const int32_t* ids, int64_t n_ids,
                                 uint16_t* out, void* stream) {
  g_msg[0] = 0;
  int rc = check_desc(desc);
  if (rc) return rc;
  if (n_ids < 0 || n_ids >= (int64_t(1) << 36)) return fail(ENGRAM_EINVAL, "bad n_ids");
  if (n_ids == 0) return ENGRAM_OK;
  if (!table || !scales || !ids || !out) return fail(ENGRAM_EINVAL, "NULL array");
  if (!aligned(table, 16) || !aligned(out, 16) || !aligned(ids, 4))
    return fail(ENGRAM_EINVAL, "table and out must be 16-byte aligned, ids 4-byte aligned");
  cudaError_t e;
  uint32_t* err = error_word(&e);
  if (!err) return cuda_fail(e, "engram_embed_rows");
  RowsArgs r{};
  r.table = table;
  r.scales = scales;
  r.ids = ids;
  r.n_ids = n_ids;
  r.num_rows = desc->num_embeddings;
  r.head_dim = desc->head_dim;
  r.out = out;
  r.err = err;
  if ((e = launch_rows(r, static_cast<cudaStream_t>(stream))) != cudaSuccess)
    return cuda_fail(e, "engram_embed_rows");
  return ENGRAM_OK;
}

ENGRAM_API int engram_embed_rows_shard(const engram_desc_t* desc, const uint8_t* table_shard,
                                       const uint8_t* scales_shard, int64_t row_begin,
                                       int64_t shard_rows, const int32_t* ids, int64_t n_ids,
                                       uint16_t* out, void* stream) {
  g_msg[0] = 0;
  int rc = check_desc(desc);
  if (rc) return rc;
  if (n_ids < 0 || n_ids >= (int64_t(1) << 36)) return fail(ENGRAM_EINVAL, "bad n_ids");
  if (row_begin < 0 || shard_rows < 0 || row_begin + shard_rows > desc->num_embeddings)
    return fail(ENGRAM_EINVAL, "the shard's rows must lie in [0, num_embeddings)");
  if (n_ids == 0) return ENGRAM_OK;
  if (!ids || !out || (shard_rows > 0 && (!table_shard || !scales_shard)))
    return fail(ENGRAM_EINVAL, "NULL array");
  if ((shard_rows > 0 && !aligned(table_shard, 16)) || !aligned(out, 16) || !aligned(ids, 4))
    return fail(ENGRAM_EINVAL, "table_shard and out must be 16-byte aligned, ids 4-byte aligned");
  cudaError_t e;
  uint32_t* err = error_word(&e);
  if (!err) return cuda_fail(e, "engram_embed_rows_shard");
  ShardRowsArgs r{};
  r.table = table_shard;
  r.scales = scales_shard;
  r.ids = ids;
  r.n_ids = n_ids;
  r.row_begin = row_begin;
  r.shard_rows = shard_rows;
  r.num_rows = desc->num_embeddings;
  r.head_dim = desc->head_dim;
  r.out = out;
  r.err = err;
  if ((e = launch_shard_rows(r, static_cast<cudaStream_t>(stream))) != cudaSuccess)
    return cuda_fail(e, "engram_embed_rows_shard");
  return ENGRAM_OK;
}

ENGRAM_API int engram_probe_stream_read(const void* src, size_t bytes, int32_t method,
                                        void* stream) {
  g_msg[0] = 0;
  if (method != kProbeBulk && method != kProbePlain && method != kProbeBulkEvictFirst)
    return fail(ENGRAM_EINVAL, "bad method");
  if (bytes % 16 != 0 || bytes >= (size_t(1) << 40))
    return fail(ENGRAM_EINVAL, "bytes must be a multiple of 16 below 2^40");
  if (bytes == 0) return ENGRAM_OK;
  if (!src || !aligned(src, 16)) return fail(ENGRAM_EINVAL, "src must be 16-byte aligned");
  cudaError_t e;
  uint32_t* err = error_word(&e);
  if (!err) return cuda_fail(e, "engram_probe_stream_read");
  if ((e = launch_stream_probe(src, static_cast<int64_t>(bytes), method, err,
                               static_cast<cudaStream_t>(stream))) != cudaSuccess)
    return cuda_fail(e, "engram_probe_stream_read");
  return ENGRAM_OK;
}

ENGRAM_API int engram_wkv(const uint16_t* a, const uint16_t* w, uint16_t* kv, int64_t M,
                          int32_t N, int32_t K, void* stream) {
  g_msg[0] = 0;
  if (M < 0 || N <= 0 || K <= 0) return fail(ENGRAM_EINVAL, "M must be >= 0, N and K > 0");
  if (M >= (int64_t(1) << 31)) return fail(ENGRAM_EINVAL, "M too large");
  if (K % 64 != 0 || N % 32 != 0)
    return fail(ENGRAM_EUNSUPPORTED, "engram_wkv needs K %% 64 == 0 and N %% 32 == 0");
  if (M == 0) return ENGRAM_OK;
  if (!a || !w || !kv) return fail(ENGRAM_EINVAL, "NULL array");
  if (!aligned(a, 16) || !aligned(w, 16) || !aligned(kv, 16))
    return fail(ENGRAM_EINVAL, "a, w and kv must be 16-byte aligned");
  if (overlaps(kv, size_t(M) * N * 2, a, size_t(M) * K * 2) ||
      overlaps(kv, size_t(M) * N * 2, w, size_t(N) * K * 2))
    return fail(ENGRAM_EINVAL, "kv overlaps an input");
  cudaError_t e;
  uint32_t* err = error_word(&e);
  if (!err) return cuda_fail(e, "engram_wkv");
  if (decode_supported(M, N, K) || small_supported(M, N, K)) {
    // few tokens: stream the weight over every SM
    WkvSmallArgs g{};
    g.a = a;
    g.w = w;
    g.kv = kv;
    g.M = M;
    g.N = N;
    g.K = K;
    g.ksplit = 1;
    g.err = err;
    e = decode_supported(M, N, K) ? launch_wkv_decode(g, static_cast<cudaStream_t>(stream))
                                  : launch_wkv_small(g, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "engram_wkv");
    return ENGRAM_OK;
  }
  WkvArgs g{a, w, kv, M, N, K, err};
  if ((e = launch_wkv(g, static_cast<cudaStream_t>(stream))) != cudaSuccess)
    return cuda_fail(e, "engram_wkv");
  return ENGRAM_OK;
}

static int gate_checks(const engram_desc_t* desc, const uint16_t* x, const uint16_t* kv,
                       const uint16_t* q, const uint16_t* k, uint16_t* out, int64_t M) {
  int rc = check_desc(desc);
  if (rc) return rc;
  if (M < 0 || M * desc->hc_mult >= (int64_t(1) << 31)) return fail(ENGRAM_EINVAL, "bad M");
  if (M == 0) return ENGRAM_OK;
  if (!x || !kv || !q || !k || !out) return fail(ENGRAM_EINVAL, "NULL array");
  if (!aligned(x, 16) || !aligned(kv, 16) || !aligned(q, 16) || !aligned(k, 16) ||
      !aligned(out, 16))
    return fail(ENGRAM_EINVAL, "x, kv, q, k and out must be 16-byte aligned");
  const size_t xbytes = size_t(M) * desc->hc_mult * desc->dim * 2;
  if (overlaps(out, xbytes, x, xbytes)) return fail(ENGRAM_EINVAL, "out overlaps x");
  return ENGRAM_OK;
}

ENGRAM_API int engram_gate_and_add(const engram_desc_t* desc, const uint16_t* x,
                                   const uint16_t* kv, const uint16_t* q_weight,
                                   const uint16_t* k_weight, const uint8_t* token_mask,
                                   uint16_t* out, float* gate_out, int64_t M, void* stream) {
  g_msg[0] = 0;
  int rc = gate_checks(desc, x, kv, q_weight, k_weight, out, M);
  if (rc || M == 0) return rc;
  GateArgs g{};
  g.x = x;
  g.kv = kv;
  g.q = q_weight;
  g.k = k_weight;
  g.mask = token_mask;
  g.out = out;
  g.gate_out = gate_out;
  g.M = M;
  g.hc = desc->hc_mult;
  g.dim = desc->dim;
  g.eps = desc->norm_eps;
  g.inv_sqrt_dim = static_cast<float>(1.0 / std::sqrt(static_cast<double>(desc->dim)));
  cudaError_t e = launch_gate(g, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "engram_gate_and_add");
  return ENGRAM_OK;
}

static FusedArgs make_fused_args(const engram_desc_t* desc, const uint16_t* rows,
                                 const uint16_t* wkv, const uint16_t* x, const uint16_t* q,
                                 const uint16_t* k, const uint8_t* mask, uint16_t* out,
                                 float* gate_out, uint16_t* kv_out, int64_t M, uint32_t* err) {
  FusedArgs f{};
  f.a = rows;
  f.w = wkv;
  f.x = x;
  f.q = q;
  f.k = k;
  f.mask = mask;
  f.out = out;
  f.gate_out = gate_out;
  f.kv_out = kv_out;
  f.M = M;
  f.K = n_hash_cols(desc) * desc->head_dim;
  f.hc = desc->hc_mult;
  f.dim = desc->dim;
  f.eps = desc->norm_eps;
  f.inv_sqrt_dim = static_cast<float>(1.0 / std::sqrt(static_cast<double>(desc->dim)));
  f.err = err;
  return f;
}

ENGRAM_API size_t engram_wkv_gate_workspace_size(const engram_desc_t* desc, int64_t M) {
  if (check_desc(desc) != ENGRAM_OK || M < 0) return 0;
  return fused_scratch_bytes(M, desc->hc_mult, desc->dim);
}

ENGRAM_API int engram_wkv_gate(const engram_desc_t* desc, const uint16_t* rows,
                               const uint16_t* wkv, const uint16_t* x, const uint16_t* q_weight,
                               const uint16_t* k_weight, const uint8_t* token_mask, uint16_t* out,
                               float* gate_out, uint16_t* kv_out, int64_t M, void* workspace,
                               size_t workspace_bytes, void* stream) {
  g_msg[0] = 0;
  int rc = gate_checks(desc, x, wkv, q_weight, k_weight, out, M);
  if (rc || M == 0) return rc;
  if (M >= (int64_t(1) << 31)) return fail(ENGRAM_EINVAL, "M too large");
  const int32_t K = n_hash_cols(desc) * desc->head_dim;
  if (!fused_supported(K, desc->hc_mult, desc->dim))
    return fail(ENGRAM_EUNSUPPORTED,
                "engram_wkv_gate needs n_hash_cols * head_dim %% 64 == 0, dim %% 256 == 0, "
                "dim <= 5120 and hc_mult <= 8; use engram_wkv + engram_gate_and_add");
  if (!rows || !aligned(rows, 16)) return fail(ENGRAM_EINVAL, "rows must be 16-byte aligned");
  if (kv_out && !aligned(kv_out, 16)) return fail(ENGRAM_EINVAL, "kv_out must be 16-byte aligned");
  const size_t need = fused_scratch_bytes(M, desc->hc_mult, desc->dim);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 256))
    return fail(ENGRAM_EINVAL, "workspace must be >= %zu bytes and 256-byte aligned", need);
  cudaError_t e;
  uint32_t* err = error_word(&e);
  if (!err) return cuda_fail(e, "engram_wkv_gate");
  FusedArgs f = make_fused_args(desc, rows, wkv, x, q_weight, k_weight, token_mask, out,
                                gate_out, kv_out, M, err);
  f.scratch = workspace;
  if ((e = launch_fused(f, static_cast<cudaStream_t>(stream))) != cudaSuccess)
    return cuda_fail(e, "engram_wkv_gate");
  return ENGRAM_OK;
}

ENGRAM_API size_t engram_forward_workspace_size(const engram_desc_t* desc, int64_t M) {
  if (check_desc(desc) != ENGRAM_OK || M < 0) return 0;
  Plan plans[kMaxPlans];
  const int n = forward_plans(desc, M, plans);
  return n > 0 ? plans[0].bytes : 0;
}

// Checks shared by the forward entry points (everything but the hash inputs); picks the fastest
// plan whose scratch fits the workspace into *plan.
static int forward_checks(const engram_desc_t* desc, const engram_weights_t* wts,
                          const uint16_t* x, uint16_t* out, uint16_t* kv_out, int64_t M,
                          void* workspace, size_t workspace_bytes, Plan* plan) {
  if (wts == nullptr) return fail(ENGRAM_EINVAL, "weights is NULL");
  int rc = gate_checks(desc, x, wts->wkv, wts->q_weight, wts->k_weight, out, M);
  if (rc || M == 0) return rc;
  if (!wts->table || !wts->scales) return fail(ENGRAM_EINVAL, "NULL table");
  if (!aligned(wts->table, 16)) return fail(ENGRAM_EINVAL, "table must be 16-byte aligned");
  if (M >= (int64_t(1) << 31)) return fail(ENGRAM_EINVAL, "B * T too large");
  const int32_t K = n_hash_cols(desc) * desc->head_dim;
  const int32_t N = desc->dim * (desc->hc_mult + 1);
  if (K % 64 != 0 || N % 32 != 0)
    return fail(ENGRAM_EUNSUPPORTED, "needs n_hash_cols * head_dim %% 64 == 0");
  if (kv_out && !aligned(kv_out, 16)) return fail(ENGRAM_EINVAL, "kv_out must be 16-byte aligned");
  Plan plans[kMaxPlans];
  const int nplans = forward_plans(desc, M, plans);
  const Plan* best = nullptr;
  size_t min_bytes = ~size_t(0);
  for (int i = 0; i < nplans; ++i) {
    if (plans[i].bytes < min_bytes) min_bytes = plans[i].bytes;
    if (best == nullptr && plans[i].bytes <= workspace_bytes) best = &plans[i];
  }
  if (workspace == nullptr || best == nullptr || !aligned(workspace, 256))
    return fail(ENGRAM_EINVAL,
                "workspace must be 256-byte aligned and >= %zu bytes (%zu for the fastest path)",
                min_bytes, nplans > 0 ? plans[0].bytes : size_t(0));
  *plan = *best;
  return ENGRAM_OK;
}

// Stages 3 + 4 of the forward by `plan`, on the gathered rows [M, K] at the start of the
// workspace (its scratch follows them). The first kernel waits, through programmatic dependent
// launch, for the kernel that wrote the rows; for the fused plan that kernel has also cleared
// the fused kernel's counters.
static int project_and_gate(const engram_desc_t* desc, const Plan& plan,
                            const engram_weights_t* wts, const uint16_t* x,
                            const uint8_t* token_mask, uint16_t* out, float* gate_out,
                            uint16_t* kv_out, int64_t M, void* workspace, const LenAdvance& adv,
                            uint32_t* err, cudaStream_t st, const char* who) {
  const int32_t K = n_hash_cols(desc) * desc->head_dim;
  const int32_t N = desc->dim * (desc->hc_mult + 1);
  const uint16_t* rows = static_cast<const uint16_t*>(workspace);
  uint8_t* ws = static_cast<uint8_t*>(workspace) + round256(size_t(M) * K * 2);
  cudaError_t e;
  if (plan.path == Path::kFused || plan.path == Path::kFusedDeferred) {
    // 3+4. projection with the gate fused into its epilogue
    FusedArgs f = make_fused_args(desc, rows, wts->wkv, x, wts->q_weight, wts->k_weight,
                                  token_mask, out, gate_out, kv_out, M, err);
    f.adv = adv;
    f.scratch = ws;
    f.sync_cleared = true;
    if (plan.path == Path::kFusedDeferred)   // value rows after the fused kernel's scratch
      f.vout = reinterpret_cast<uint16_t*>(ws + round256(fused_scratch_bytes(M, desc->hc_mult,
                                                                              desc->dim)));
    if ((e = launch_fused(f, st, true)) != cudaSuccess) return cuda_fail(e, who, "fused");
    if (plan.path == Path::kFusedDeferred) {
      GateApplyArgs g{};
      g.x = x;
      g.gx = fused_gates(ws);
      g.value = f.vout;
      g.mask = token_mask;
      g.out = out;
      g.M = M;
      g.hc = desc->hc_mult;
      g.dim = desc->dim;
      if ((e = launch_gate_apply(g, st, true)) != cudaSuccess)
        return cuda_fail(e, who, "gate apply");
    }
    return ENGRAM_OK;
  }
  // 3. projection -> bf16 kv (or f32 split-K partials); 4. gate and add
  GateArgs ga{};
  if (plan.path == Path::kDecode) {
    WkvSmallArgs g{};
    g.a = rows;
    g.w = wts->wkv;
    g.kv = kv_out ? kv_out : reinterpret_cast<uint16_t*>(ws);
    g.M = M;
    g.N = N;
    g.K = K;
    g.ksplit = 1;
    g.err = err;
    if ((e = launch_wkv_decode(g, st, true)) != cudaSuccess) return cuda_fail(e, who, "wkv");
    ga.kv = g.kv;
  } else if (plan.path == Path::kSmall) {
    WkvSmallArgs g{};
    g.a = rows;
    g.w = wts->wkv;
    g.M = M;
    g.N = N;
    g.K = K;
    g.ksplit = plan.ksplit;
    g.err = err;
    if (plan.ksplit > 1) {
      g.part = reinterpret_cast<float*>(ws);
      ga.part = g.part;
      ga.ksplit = plan.ksplit;
      ga.kv_out = kv_out;
    } else {
      g.kv = kv_out ? kv_out : reinterpret_cast<uint16_t*>(ws);
      ga.kv = g.kv;
    }
    if ((e = launch_wkv_small(g, st, true)) != cudaSuccess) return cuda_fail(e, who, "wkv");
  } else {
    uint16_t* kv = kv_out ? kv_out : reinterpret_cast<uint16_t*>(ws);
    WkvArgs g{rows, wts->wkv, kv, M, N, K, err};
    if ((e = launch_wkv(g, st, true)) != cudaSuccess) return cuda_fail(e, who, "wkv");
    ga.kv = kv;
  }
  ga.x = x;
  ga.q = wts->q_weight;
  ga.k = wts->k_weight;
  ga.mask = token_mask;
  ga.out = out;
  ga.gate_out = gate_out;
  ga.M = M;
  ga.hc = desc->hc_mult;
  ga.dim = desc->dim;
  ga.eps = desc->norm_eps;
  ga.inv_sqrt_dim = static_cast<float>(1.0 / std::sqrt(static_cast<double>(desc->dim)));
  ga.adv = adv;
  if ((e = launch_gate(ga, st, true)) != cudaSuccess) return cuda_fail(e, who, "gate");
  return ENGRAM_OK;
}

ENGRAM_API int engram_forward(const engram_desc_t* desc, const engram_tables_t* tables,
                              const engram_weights_t* wts, const uint16_t* x,
                              const int32_t* tokens, int32_t B, int32_t T, int32_t* cache,
                              int32_t* cache_len, int32_t capacity, const uint8_t* token_mask,
                              uint16_t* out, int32_t* hash_ids_out, float* gate_out,
                              uint16_t* kv_out, void* workspace, size_t workspace_bytes,
                              void* stream) {
  g_msg[0] = 0;
  int rc = hash_checks(desc, tables, tokens, B, T, cache, cache_len, capacity, hash_ids_out,
                       /*ids_optional=*/true);
  if (rc) return rc;
  const int64_t M = int64_t(B) * T;
  Plan plan{};
  rc = forward_checks(desc, wts, x, out, kv_out, M, workspace, workspace_bytes, &plan);
  if (rc || M == 0) return rc;
  cudaError_t e;
  uint32_t* err = error_word(&e);
  if (!err) return cuda_fail(e, "engram_forward");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint16_t* rows = static_cast<uint16_t*>(workspace);   // the projection's input [M, K]
  HashArgs h = make_hash_args(desc, tables, tokens, B, T, cache, cache_len, capacity,
                              hash_ids_out, err);
  HashRowsArgs hr = single_layer_hash_rows(h, wts->table, wts->scales, desc->num_embeddings,
                                           desc->head_dim, rows);
  // 1+2. hash every slot and gather its row into the projection's input, in one kernel. The
  // kernels of the chain are launched with programmatic stream serialization: each overlaps its
  // launch and prologue with the previous one and waits for it before touching its data.
  const int32_t K = n_hash_cols(desc) * desc->head_dim;
  // the fused kernel's counters, cleared by the hash kernel
  if (plan.path == Path::kFused || plan.path == Path::kFusedDeferred)
    fused_sync_region(static_cast<uint8_t*>(workspace) + round256(size_t(M) * K * 2), M,
                      desc->hc_mult, desc->dim, &hr.zero, &hr.zero_n);
  if ((e = launch_hash_rows(hr, st, true)) != cudaSuccess)
    return cuda_fail(e, "engram_forward: hash + rows");
  // 3+4; the kernel that runs last advances the cache lengths (every reader of them is done)
  const LenAdvance adv{cache_len, B, T, capacity};
  return project_and_gate(desc, plan, wts, x, token_mask, out, gate_out, kv_out, M, workspace,
                          adv, err, st, "engram_forward");
}

ENGRAM_API int engram_forward_ids(const engram_desc_t* desc, const engram_weights_t* wts,
                                  const uint16_t* x, const int32_t* hash_ids, int64_t M,
                                  const uint8_t* token_mask, uint16_t* out, float* gate_out,
                                  uint16_t* kv_out, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  g_msg[0] = 0;
  int rc = check_desc(desc);
  if (rc) return rc;
  if (M < 0) return fail(ENGRAM_EINVAL, "M must be >= 0");
  Plan plan{};
  rc = forward_checks(desc, wts, x, out, kv_out, M, workspace, workspace_bytes, &plan);
  if (rc || M == 0) return rc;
  if (hash_ids == nullptr || !aligned(hash_ids, 4))
    return fail(ENGRAM_EINVAL, "hash_ids must be a 4-byte aligned device array");
  const int S = n_hash_cols(desc);
  const int32_t K = S * desc->head_dim;
  if (overlaps(hash_ids, size_t(M) * S * 4, workspace, round256(size_t(M) * K * 2)))
    return fail(ENGRAM_EINVAL, "hash_ids overlaps the workspace");
  cudaError_t e;
  uint32_t* err = error_word(&e);
  if (!err) return cuda_fail(e, "engram_forward_ids");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // 2. gather and dequantise the rows of every id into the projection's input
  RowsArgs r{};
  r.table = wts->table;
  r.scales = wts->scales;
  r.ids = hash_ids;
  r.n_ids = M * S;
  r.num_rows = desc->num_embeddings;
  r.head_dim = desc->head_dim;
  r.out = static_cast<uint16_t*>(workspace);
  r.err = err;
  // the fused kernel's counters, cleared by the rows kernel
  if (plan.path == Path::kFused || plan.path == Path::kFusedDeferred)
    fused_sync_region(static_cast<uint8_t*>(workspace) + round256(size_t(M) * K * 2), M,
                      desc->hc_mult, desc->dim, &r.zero, &r.zero_n);
  if ((e = launch_rows(r, st, true)) != cudaSuccess)
    return cuda_fail(e, "engram_forward_ids: rows");
  const LenAdvance adv{nullptr, 0, 0, 0};
  return project_and_gate(desc, plan, wts, x, token_mask, out, gate_out, kv_out, M, workspace,
                          adv, err, st, "engram_forward_ids");
}

}  // extern "C"
