/*
 * engram.h - C ABI of the GB300 (sm_103a) Engram forward path of DeepSeek V4.1.
 *
 * The path has four stages (page "Module engram", CPU reference, stage list 1-4):
 *   1. hash        token ids -> 24 table-row ids per position, through an n-gram hash whose
 *                  look-back cache spans calls (prefill then decode);
 *   2. embed_rows  gather those rows from an fp8 e4m3 table and dequantise them by e8m0 block
 *                  scales to bf16;
 *   3. wkv         one bf16 projection [24 * head_dim] -> [dim * (hc_mult + 1)], f32 accumulate,
 *                  bf16 output: hc_mult keys (one per residual stream) and one shared value;
 *   4. gate_and_add  per (token, stream): a normalised dot of the stream with its key, weighted by
 *                  q_weight * k_weight, a signed-sqrt sigmoid gate, and stream + gate * value
 *                  rounded to bf16.
 * Each stage has its own entry point; engram_forward runs all four.
 *
 * Conventions for every entry point:
 *  - All array pointers are DEVICE pointers owned by the caller; the library allocates no device
 *    memory on these calls. Scratch memory is caller-provided (engram_forward_workspace_size).
 *  - Arrays are dense, row-major, contiguous. bf16 values travel as uint16_t bit patterns, fp8
 *    e4m3fn and e8m0 as uint8_t. Every array pointer must be 16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Work is enqueued
 *    asynchronously; a return of ENGRAM_OK means "validated and launched", not "finished".
 *  - Return value: an engram_status. Arguments are validated on the host before anything is
 *    launched: a bad argument returns ENGRAM_EINVAL (or ENGRAM_EUNSUPPORTED for a shape the
 *    kernels do not cover) and launches nothing. Problems that only the device can see (a token
 *    id outside the vocabulary, a hash id outside the table, a full cache, a kernel wait that gave
 *    up) set bits in a device error word; engram_check_errors synchronises `stream`, reads the
 *    word, clears it and returns ENGRAM_EDEVICE (or ENGRAM_ECAPACITY for a full cache).
 *  - engram_last_error() gives a message for the last non-OK return on the calling thread.
 *  - Calls that are in flight at the same time on different streams must not share output or
 *    cache buffers.
 *  - Calls may come from several host threads and for several devices (each call runs on the
 *    device current on its thread). The library's host-side state (the device error word, SM
 *    counts, kernel attributes) is kept per device and guarded; the error word is shared by all
 *    calls on one device.
 *  - That per-device state (including the device addresses of the error word and of
 *    engram_forward_noalloc's scratch) is looked up once and kept for the life of the process.
 *    cudaDeviceReset unloads the library's device code and invalidates it: do not use the
 *    library on a device after resetting it.
 */
#ifndef ENGRAM_H_
#define ENGRAM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ENGRAM_API __attribute__((visibility("default")))

typedef enum engram_status {
  ENGRAM_OK = 0,
  ENGRAM_EINVAL = 1,       /* bad argument: NULL, negative size, misaligned, aliasing, geometry */
  ENGRAM_ECAPACITY = 2,    /* a look-back cache ran out of capacity (device-detected)        */
  ENGRAM_ECUDA = 3,        /* a CUDA runtime call or launch failed                             */
  ENGRAM_EDEVICE = 4,      /* the device error word was set (see engram_check_errors)         */
  ENGRAM_EUNSUPPORTED = 5  /* valid, but outside the shapes these kernels implement           */
} engram_status;

/* Device error word bits, as returned through engram_check_errors(..., &bits). */
#define ENGRAM_DEVERR_TOKEN_RANGE 1u    /* token id outside [0, vocab)            */
#define ENGRAM_DEVERR_CACHE_FULL 2u     /* cache_len + T > capacity                */
#define ENGRAM_DEVERR_ID_RANGE 4u       /* hash id outside [0, num_embeddings)     */
#define ENGRAM_DEVERR_WAIT_TIMEOUT 8u   /* a bounded in-kernel wait gave up        */

/*
 * Geometry of one Engram layer (Engram listing, __init__: dim, hc_mult, the layout's n_heads,
 * max_ngram_size, head_dim and num_embeddings; norm_eps is ModelArgs.norm_eps, whose value the
 * pages do not give). n_hash_cols = (max_ngram_size - 1) * n_heads rows are fetched per position.
 * Requirements: all sizes > 0; 2 <= max_ngram_size <= 8; head_dim % 32 == 0 (one e8m0 scale per 32
 * elements); dim % 8 == 0; num_embeddings < 2^31; norm_eps >= 0.
 */
typedef struct engram_desc {
  int32_t dim;
  int32_t hc_mult;
  int32_t n_heads;
  int32_t max_ngram_size;
  int32_t head_dim;
  int32_t reserved;
  int64_t num_embeddings;
  float norm_eps;
} engram_desc_t;

/*
 * Hash tables, consumed as given (page "Module engram": the tables paragraph and struct
 * EngramTables). All pointers are device pointers.
 *   token_map   int32 [vocab]: tokenizer id -> compressed id (>= 0).
 *   pad_id      compressed id that fills a window before the sequence start (>= 0).
 *   multipliers uint64 [max_ngram_size]: multiplier m_k of look-back k (k = 0 is the current
 *               position); shared by every n-gram size and head.
 *   primes      uint64 [n_hash_cols]: modulus P_s of slot s = (n - 2) * n_heads + head.
 *   offsets     int64 [n_hash_cols]: first table row O_s of slot s.
 * Slot s of position p: id = (mix_n mod P_s) + O_s with mix_n = XOR_{k<n} (c_{p-k} * m_k), all on
 * unsigned 64-bit words (multiply wraps modulo 2^64).
 */
typedef struct engram_tables {
  const int32_t* token_map;
  int32_t vocab;
  int32_t pad_id;
  const uint64_t* multipliers;
  const uint64_t* primes;
  const int64_t* offsets;
} engram_tables_t;

/*
 * Parameters of one Engram layer (Engram listing, __init__: embed, wkv, q_weight, k_weight).
 *   table    uint8 e4m3fn [num_embeddings, head_dim]      (ParallelEngramEmbedding values)
 *   scales   uint8 e8m0   [num_embeddings, head_dim / 32] (one power-of-two scale per 32 values)
 *   wkv      bf16 [dim * (hc_mult + 1), n_hash_cols * head_dim]  (Linear weight, [out, in])
 *   q_weight bf16 [hc_mult, dim];  k_weight bf16 [hc_mult, dim]
 */
typedef struct engram_weights {
  const uint8_t* table;
  const uint8_t* scales;
  const uint16_t* wkv;
  const uint16_t* q_weight;
  const uint16_t* k_weight;
} engram_weights_t;

/*
 * One Engram layer's part in engram_hash_rows_layers. Each Engram layer takes its own entry of the
 * hash layout (Engram listing, __init__: layer_hash_index = the layer's place in
 * layout.layer_ids; its embedding has layout.num_embeddings[layer_hash_index] rows), so it has its
 * own hash constants and table. All pointers are device pointers.
 *   multipliers uint64 [max_ngram_size], primes uint64 [n_hash_cols], offsets int64 [n_hash_cols]:
 *                  this layer's constants, with the meaning they have in engram_tables_t;
 *   num_embeddings rows of this layer's table, in [1, 2^31);
 *   table uint8 e4m3fn [num_embeddings, head_dim] (16-byte aligned), scales uint8 e8m0
 *                  [num_embeddings, head_dim / 32]: this layer's embedding, as in engram_weights_t;
 *   rows     out: bf16 [B * T, n_hash_cols * head_dim] (16-byte aligned), the layer's gathered and
 *                  dequantised rows, i.e. the rows argument of engram_wkv_gate for this layer;
 *   hash_ids out: int32 [B * T, n_hash_cols], or NULL.
 */
typedef struct engram_layer_hash {
  const uint64_t* multipliers;
  const uint64_t* primes;
  const int64_t* offsets;
  int64_t num_embeddings;
  const uint8_t* table;
  const uint8_t* scales;
  uint16_t* rows;
  int32_t* hash_ids;
} engram_layer_hash_t;

#define ENGRAM_MAX_HASH_LAYERS 16

/* Message for the last non-OK status returned on this thread ("" if none). Never NULL. */
ENGRAM_API const char* engram_last_error(void);

/* Library ABI version (ENGRAM_ABI_VERSION). */
#define ENGRAM_ABI_VERSION 1
ENGRAM_API int32_t engram_abi_version(void);

/*
 * Synchronise `stream`, read and clear the device error word. Returns ENGRAM_OK if it was clear,
 * ENGRAM_ECAPACITY if only the cache-full bit was set, ENGRAM_EDEVICE otherwise, ENGRAM_ECUDA if
 * the synchronisation itself failed. `bits_out` (host pointer, may be NULL) receives the word.
 */
ENGRAM_API int engram_check_errors(void* stream, uint32_t* bits_out);

/*
 * Stage 1, the n-gram hash (page "Module engram", stage 1 Hash and struct NgramHashState).
 *   tokens     int32 [B, T]          token ids of this call (T new positions per sequence).
 *   cache      int32 [B, capacity]   compressed ids of every position seen so far (in/out).
 *   cache_len  int32 [B]             positions already in each sequence's cache (in/out: += T).
 *   hash_ids   int32 [B, T, n_hash_cols]  out.
 * Position t of sequence b is absolute position p = cache_len[b] + t; its window reaches back
 * into the cache, so a decode step (T = 1) sees the prefill. Before position 0 the window holds
 * pad_id. A token outside [0, vocab) is hashed as pad_id and sets ENGRAM_DEVERR_TOKEN_RANGE; a
 * sequence whose cache would exceed `capacity` sets ENGRAM_DEVERR_CACHE_FULL and the positions
 * beyond capacity are not cached. B = 0 or T = 0 launches nothing.
 */
ENGRAM_API int engram_hash(const engram_desc_t* desc, const engram_tables_t* tables,
                           const int32_t* tokens, int32_t B, int32_t T, int32_t* cache,
                           int32_t* cache_len, int32_t capacity, int32_t* hash_ids,
                           void* stream);

/*
 * Stage 2, table rows (page "Module engram", stage 2 and function embed_rows; Engram listing,
 * forward: self.embed(hash_ids)). out[i, d] = bf16(e4m3(table[ids[i], d]) *
 * 2^(scales[ids[i], d / 32] - 127)); exact for every scale that keeps the product a normal bf16.
 *   ids  int32 [n_ids];  out bf16 [n_ids, head_dim].
 * An id outside [0, num_embeddings) writes a zero row and sets ENGRAM_DEVERR_ID_RANGE.
 */
ENGRAM_API int engram_embed_rows(const engram_desc_t* desc, const uint8_t* table,
                                 const uint8_t* scales, const int32_t* ids, int64_t n_ids,
                                 uint16_t* out, void* stream);

/*
 * Stage 2 over a row-sharded table (Engram listing, __init__: the embedding is a
 * ParallelEngramEmbedding; the pages do not say how it splits the table: this library reads it
 * as contiguous ranges of rows, one per rank). The calling rank holds rows
 * [row_begin, row_begin + shard_rows) of the num_embeddings-row table:
 *   table_shard uint8 e4m3fn [shard_rows, head_dim] (16-byte aligned), scales_shard uint8 e8m0
 *   [shard_rows, head_dim / 32]; ids int32 [n_ids] GLOBAL row ids; out bf16 [n_ids, head_dim].
 * A row the rank holds is written as engram_embed_rows writes it; a row in [0, num_embeddings)
 * that another rank holds is written as bf16 -0.0 in every element. -0 is the identity of IEEE
 * addition, so the element-wise bf16 sum of every rank's out (an all-reduce, in any order) equals
 * engram_embed_rows over the whole table bit for bit, signed zeros included. An id outside
 * [0, num_embeddings) writes a zero row and sets ENGRAM_DEVERR_ID_RANGE (on every rank).
 * A shard outside [0, num_embeddings) returns ENGRAM_EINVAL; shard_rows = 0 (a rank with no rows)
 * writes -0 rows only. The exchange itself is the caller's (one all-reduce of out).
 */
ENGRAM_API int engram_embed_rows_shard(const engram_desc_t* desc, const uint8_t* table_shard,
                                       const uint8_t* scales_shard, int64_t row_begin,
                                       int64_t shard_rows, const int32_t* ids, int64_t n_ids,
                                       uint16_t* out, void* stream);

/*
 * Stage 3, the wkv projection (page "Module engram", stage 3 and function linear_bf16; Engram
 * listing, forward: self.wkv(...)). kv[m, n] = bf16(sum_k a[m, k] * w[n, k]), f32 accumulation
 * on the tensor cores, one rounding to bf16.
 *   a bf16 [M, K];  w bf16 [N, K];  kv bf16 [M, N].
 * Requires K % 64 == 0 and N % 32 == 0 (else ENGRAM_EUNSUPPORTED). M = 0 launches nothing.
 */
ENGRAM_API int engram_wkv(const uint16_t* a, const uint16_t* w, uint16_t* kv, int64_t M,
                          int32_t N, int32_t K, void* stream);

/*
 * Stage 4, gate and add (page "Module engram", function gate_and_add; Engram listing, forward
 * after the projection; page "DeepSeek V4.1 · Gate per stream", formulas for a_k and g^e_k).
 * For token m and stream s, with h = x[m, s, :], key = kv[m, s*dim : (s+1)*dim],
 * value = kv[m, hc*dim : (hc+1)*dim] and w = q_weight[s] * k_weight[s]:
 *   a = sum(h * w * key) / (sqrt(mean(h^2) + eps) * sqrt(mean(key^2) + eps) * sqrt(dim))
 *   gate = sigmoid(copysign(sqrt(max(|a|, 1e-6)), a)), or 0 where token_mask[m] == 0
 *   out[m, s, :] = bf16(h + gate * value)
 * A masked token's row is written as an exact copy of x.
 *   x bf16 [M, hc, dim]; kv bf16 [M, dim * (hc + 1)]; q_weight, k_weight bf16 [hc, dim];
 *   token_mask uint8 [M] (nonzero = keep the gate) or NULL (all kept);
 *   out bf16 [M, hc, dim] (must not overlap x); gate_out f32 [M, hc] or NULL.
 */
ENGRAM_API int engram_gate_and_add(const engram_desc_t* desc, const uint16_t* x,
                                   const uint16_t* kv, const uint16_t* q_weight,
                                   const uint16_t* k_weight, const uint8_t* token_mask,
                                   uint16_t* out, float* gate_out, int64_t M, void* stream);

/*
 * Stages 1 + 2 for several Engram layers in one launch (page "Module engram", stages 1 and 2;
 * Engram listing, __init__: layer_hash_index; forward: self.embed(hash_ids)). A model's Engram
 * layers all hash the same token stream: the window of compressed ids of each position (token
 * map, look-back cache, pad) is resolved once and shared; each layer then forms its own slot ids
 * with its own constants and gathers + dequantises its own rows, exactly as engram_hash followed
 * by engram_embed_rows would for that layer. The cache is appended and cache_len advanced once
 * (by T), as one engram_hash call would. Each layer's rows then feed engram_wkv_gate (or
 * engram_wkv + engram_gate_and_add) with that layer's x.
 *   desc: the geometry shared by the layers (n_heads, max_ngram_size, head_dim; num_embeddings
 *         is not read, each layer gives its own);
 *   tables: token_map, vocab and pad_id are used; multipliers, primes and offsets are not read
 *           (they may be NULL);
 *   layers: host array of n_layers (1 .. ENGRAM_MAX_HASH_LAYERS) layer records, read during the
 *           call only; tokens, cache, cache_len, capacity as in engram_hash.
 * Errors: as engram_hash and engram_embed_rows (an id outside a layer's [0, num_embeddings)
 * writes a zero row and sets ENGRAM_DEVERR_ID_RANGE); n_layers out of range, a NULL or
 * misaligned layer pointer, or outputs that overlap the cache return ENGRAM_EINVAL. B = 0 or
 * T = 0 launches nothing.
 */
ENGRAM_API int engram_hash_rows_layers(const engram_desc_t* desc, const engram_tables_t* tables,
                                       const engram_layer_hash_t* layers, int32_t n_layers,
                                       const int32_t* tokens, int32_t B, int32_t T,
                                       int32_t* cache, int32_t* cache_len, int32_t capacity,
                                       void* stream);

/*
 * Stages 3 + 4 in one tensor-core kernel (Engram listing, forward: self.wkv(...) followed by the
 * gate and add): the projection of already-gathered rows with the gate-and-add in its epilogue,
 * so the kv row is never written to memory (unless kv_out is given).
 *   rows bf16 [M, n_hash_cols * head_dim] (the output of engram_embed_rows, flattened per token);
 *   wkv bf16 [dim * (hc + 1), n_hash_cols * head_dim]; x, q_weight, k_weight, token_mask, out,
 *   gate_out as in engram_gate_and_add; kv_out bf16 [M, dim * (hc + 1)] or NULL;
 *   workspace: device scratch of at least engram_wkv_gate_workspace_size(desc, M) bytes,
 *   256-byte aligned, not shared with a concurrent call (per-column-tile partial sums of the
 *   gate, the gates, and the counters and flags the CTAs coordinate through; the counters are
 *   cleared on the stream before each launch, so nothing in it needs to start at zero).
 * The kernel is persistent (one CTA per SM) but does not need all of its CTAs resident at once:
 * CTAs take work in an order in which everything a CTA waits for is held by a running CTA.
 * Results equal engram_wkv followed by engram_gate_and_add up
 * to f32 summation order in the gate, and are the same from run to run. Requires
 * n_hash_cols * head_dim % 64 == 0, dim % 256 == 0, dim <= 5120 and hc_mult <= 8; otherwise
 * returns ENGRAM_EUNSUPPORTED (use the two separate calls).
 */
ENGRAM_API size_t engram_wkv_gate_workspace_size(const engram_desc_t* desc, int64_t M);
ENGRAM_API int engram_wkv_gate(const engram_desc_t* desc, const uint16_t* rows,
                               const uint16_t* wkv, const uint16_t* x, const uint16_t* q_weight,
                               const uint16_t* k_weight, const uint8_t* token_mask, uint16_t* out,
                               float* gate_out, uint16_t* kv_out, int64_t M, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * Bytes of scratch for engram_forward on M = B * T tokens with the fastest projection path (a
 * multiple of 256). engram_forward also accepts a smaller workspace and then runs the fastest
 * path that fits it; the smallest it accepts holds the gathered rows and the fused kernel's
 * scratch (4,048 bytes per token at the full geometry, plus 64 bytes per 256 tokens and 4 bytes,
 * each part rounded up to a multiple of 256).
 */
ENGRAM_API size_t engram_forward_workspace_size(const engram_desc_t* desc, int64_t M);

/*
 * The whole Engram forward (Engram listing, forward; page "Module engram", stages 1-4) for B
 * sequences of T new tokens each: hash with the look-back cache, gather and dequantise rows,
 * project, gate and add. Arguments as in the stage calls above, plus
 *   x bf16 [B, T, hc, dim]; token_mask uint8 [B, T] or NULL; out bf16 [B, T, hc, dim];
 *   hash_ids_out int32 [B, T, n_hash_cols] or NULL; gate_out f32 [B, T, hc] or NULL;
 *   kv_out bf16 [B, T, dim * (hc + 1)] or NULL (the projection, for inspection; costs traffic);
 *   workspace: device scratch, 256-byte aligned, not shared with a concurrent call; see
 *   engram_forward_workspace_size for its size.
 * How stages 3 and 4 run depends on M and on the workspace given (the fastest path that fits):
 * up to 256 tokens, a weight-streaming projection over every SM (for up to 64 tokens, a fixed
 * share of the weight rows per SM) into a bf16 kv, then the gate kernel; below 512 tokens, the
 * persistent projection GEMM into a bf16 kv then the gate kernel; from 240 to 256 and from 512
 * to 2048 tokens, the fused projection kernel with its output deferred (it computes the gates and
 * stores the bf16 value rows; a second kernel then writes out = x + gate * value), bit for bit
 * what the fused kernel gives; above 2048 tokens, or when only the minimum workspace is given,
 * the projection with the gate fused into its epilogue (as engram_wkv_gate). Every path runs on
 * the GPU; results agree within the projection's f32-summation bound.
 */
ENGRAM_API int engram_forward(const engram_desc_t* desc, const engram_tables_t* tables,
                              const engram_weights_t* weights, const uint16_t* x,
                              const int32_t* tokens, int32_t B, int32_t T, int32_t* cache,
                              int32_t* cache_len, int32_t capacity, const uint8_t* token_mask,
                              uint16_t* out, int32_t* hash_ids_out, float* gate_out,
                              uint16_t* kv_out, void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * Stages 2-4 from hash ids computed elsewhere: the Engram listing's forward(x, hash_ids,
 * token_mask) itself (Engram listing, forward; page "Module engram", stages 2-4). Gathers and
 * dequantises the rows of hash_ids, projects, gates and adds, through the same token-count
 * dependent paths as engram_forward (the ids may come from engram_hash, from
 * engram_hash_rows_layers' hash_ids, or from the caller's own hash).
 *   hash_ids int32 [M, n_hash_cols] (device, 4-byte aligned, not overlapping the workspace);
 *   x bf16 [M, hc, dim]; token_mask uint8 [M] or NULL; out, gate_out, kv_out as in
 *   engram_forward; workspace as in engram_forward (engram_forward_workspace_size(desc, M) bytes
 *   for the fastest path, at least the same minimum).
 * An id outside [0, num_embeddings) gathers a zero row and sets ENGRAM_DEVERR_ID_RANGE. M = 0
 * launches nothing.
 */
ENGRAM_API int engram_forward_ids(const engram_desc_t* desc, const engram_weights_t* weights,
                                  const uint16_t* x, const int32_t* hash_ids, int64_t M,
                                  const uint8_t* token_mask, uint16_t* out, float* gate_out,
                                  uint16_t* kv_out, void* workspace, size_t workspace_bytes,
                                  void* stream);

/*
 * engram_forward without a workspace argument, for callers that cannot allocate device memory
 * (a runtime that owns all device memory and passes a plugin only its inputs and outputs, or a
 * serving loop that must not call cudaMalloc, which can synchronise the device). The pages have
 * no counterpart of this call; it exists for the callers just named.
 *
 * Arguments and results are those of engram_forward. The scratch (hash ids and gathered rows)
 * lives in a fixed array of ENGRAM_NOALLOC_SCRATCH_BYTES (8 MiB) that the library keeps in every
 * GPU that loads it, until the process exits. A call whose scratch would not fit returns
 * ENGRAM_EINVAL and launches nothing: at the full geometry (dim 5120, hc 4, 24 rows of
 * head_dim 64) that is more than 2,048 tokens (B * T) per call. Within that limit the call runs
 * the fastest projection path whose scratch fits in the array.
 *
 * This call allocates nothing: no cudaMalloc, no cudaFree, no allocating library routine. Its
 * first call on a device looks up the array's device address (cudaGetSymbolAddress, with that
 * device current) and keeps it for the life of the process. Every call shares the one
 * array and leaves its contents behind; nothing in it needs to start at zero, since each call
 * writes all of the scratch it reads. Calls whose work overlaps on the GPU (different streams,
 * or host threads) race on the array: serialise them.
 */
#define ENGRAM_NOALLOC_SCRATCH_BYTES (8 * 1024 * 1024)
ENGRAM_API int engram_forward_noalloc(const engram_desc_t* desc, const engram_tables_t* tables,
                                      const engram_weights_t* weights, const uint16_t* x,
                                      const int32_t* tokens, int32_t B, int32_t T, int32_t* cache,
                                      int32_t* cache_len, int32_t capacity,
                                      const uint8_t* token_mask, uint16_t* out,
                                      int32_t* hash_ids_out, float* gate_out, uint16_t* kv_out,
                                      void* stream);

/*
 * The whole forward of engram_forward as one CUDA graph that the library builds and owns, for
 * loops that run the same step shape again and again (decode: B sequences, T = 1 each step).
 * engram_forward_graph_create takes engram_forward's arguments (without the stream), validates
 * them as engram_forward does, captures engram_forward's kernel chain on a private stream (no
 * kernel runs at creation) and instantiates it; *graph_out receives the handle, NULL on error.
 * engram_graph_launch replays it on `stream` (one graph launch: the hash + gather, projection
 * and gate kernels with their programmatic dependent launches), exactly as one engram_forward
 * call with the creation's arguments would run. Every pointer given at creation is baked in:
 * refill x, tokens and token_mask in place before each launch; the cache and cache_len advance
 * on the device with every launch, as with consecutive engram_forward calls; out, gate_out,
 * hash_ids_out, kv_out and the workspace are rewritten by every launch. Launches of one graph
 * must not overlap each other or other work on the same buffers (they share the workspace).
 * The graph belongs to the device current at creation; launching it with another device current
 * returns ENGRAM_EINVAL. engram_graph_destroy frees it (NULL is allowed); destroy it before the
 * buffers it names are freed. Errors: as engram_forward; a failed capture or instantiation
 * returns ENGRAM_ECUDA.
 */
typedef struct engram_graph engram_graph_t;
ENGRAM_API int engram_forward_graph_create(
    const engram_desc_t* desc, const engram_tables_t* tables, const engram_weights_t* weights,
    const uint16_t* x, const int32_t* tokens, int32_t B, int32_t T, int32_t* cache,
    int32_t* cache_len, int32_t capacity, const uint8_t* token_mask, uint16_t* out,
    int32_t* hash_ids_out, float* gate_out, uint16_t* kv_out, void* workspace,
    size_t workspace_bytes, engram_graph_t** graph_out);
ENGRAM_API int engram_graph_launch(const engram_graph_t* graph, void* stream);
ENGRAM_API int engram_graph_destroy(engram_graph_t* graph);

/*
 * A measurement call, not a stage of the forward (it has no counterpart on the pages): one read of
 * the device buffer src[0, bytes) spread evenly over every SM, discarding the bytes. Its duration
 * bounds from below any kernel that streams the same buffer once from the same memory state (the
 * decode projection streams the wkv weight once per step), whatever that kernel computes.
 *   method 0: 32 KB bulk copies (cp.async.bulk) into a 6-stage shared-memory ring per SM (the
 *             decode projection's bytes in flight); method 1: 16-byte non-caching loads, 512
 *             threads per SM, four loads in flight per thread; method 2: as method 0, with an L2
 *             evict-first policy on the copies (the decode projection's policy for the weight).
 * src must be 16-byte aligned and bytes a multiple of 16 (else ENGRAM_EINVAL); bytes = 0 launches
 * nothing. Writes nothing the caller can see.
 */
ENGRAM_API int engram_probe_stream_read(const void* src, size_t bytes, int32_t method,
                                        void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ENGRAM_H_ */
