// Memory-bound stages of the Engram forward: the n-gram hash (stage 1), the fp8 row gather and
// dequantisation (stage 2) and the standalone gate-and-add (stage 4).
#include "device.cuh"
#include "hash_rows.cuh"
#include "kernels.h"

namespace engram {

// ------------------------------------------------------------------------------ stage 1: hash
// Page "Module engram", stage 1 and struct NgramHashState. One thread per (position, slot).
// Slot s belongs to n-gram size n = s / n_heads + 2; its window is c_{p-k}, k = 0..n-1, taken
// from this call's tokens (k <= t), from the cache (earlier calls), or pad_id (before p = 0).

// Hash id of flat work item i = (b, t, s); appends c_p to the cache when s == 0.
__device__ __forceinline__ int32_t hash_slot(const HashArgs& a, int64_t i) {
  const int32_t S = (a.max_ngram - 1) * a.n_heads;
  const int32_t s = static_cast<int32_t>(i % S);
  const int64_t bt = i / S;
  const int32_t t = static_cast<int32_t>(bt % a.T);
  const int32_t b = static_cast<int32_t>(bt / a.T);
  const int32_t n = s / a.n_heads + 2;
  const int32_t len0 = a.cache_len[b];

  uint64_t mix = 0;
  int32_t c0 = 0;
  for (int32_t k = 0; k < n; ++k) {
    const int32_t c = compressed_id(a, b, t, len0, k);
    if (k == 0) c0 = c;
    mix ^= static_cast<uint64_t>(static_cast<int64_t>(c)) * __ldg(a.multipliers + k);
  }
  const uint64_t P = __ldg(a.primes + s);
  const int32_t id = static_cast<int32_t>(static_cast<int64_t>(mix % P) + __ldg(a.offsets + s));

  if (s == 0) {  // one thread per position appends c_p to the cache
    const int64_t p = static_cast<int64_t>(len0) + t;
    if (p < a.capacity) {
      a.cache[static_cast<int64_t>(b) * a.capacity + p] = c0;
    } else {
      set_error(a.err, kErrCacheCapacity);
    }
  }
  return id;
}

__global__ void __launch_bounds__(256) hash_kernel(HashArgs a) {
  const int32_t S = (a.max_ngram - 1) * a.n_heads;
  const int64_t total = static_cast<int64_t>(a.B) * a.T * S;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= total) return;
  a.hash_ids[i] = hash_slot(a, i);
}

__global__ void advance_len_kernel(int32_t* len, int32_t B, int32_t T, int32_t cap) {
  const int32_t b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) len[b] = min(len[b] + T, cap);
}

cudaError_t launch_hash(const HashArgs& a, cudaStream_t st) {
  const int64_t S = (a.max_ngram - 1) * a.n_heads;
  const int64_t total = static_cast<int64_t>(a.B) * a.T * S;
  const int64_t blocks = (total + 255) / 256;
  hash_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_advance_len(int32_t* len, int32_t B, int32_t T, int32_t cap, cudaStream_t st) {
  advance_len_kernel<<<(B + 255) / 256, 256, 0, st>>>(len, B, T, cap);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------ stage 2: table rows
// Page "Module engram", stage 2 / embed_rows / regen_table: value * scale per 32-block, to bf16.

__global__ void __launch_bounds__(256) rows_kernel(RowsArgs a) {
  pdl_wait();   // the ids may come from the previous kernel of the stream
  pdl_launch_dependents();
  // the next kernel's counters (it reads them only after this grid has completed)
  if (a.zero != nullptr && blockIdx.x == 0)
    for (int32_t i = threadIdx.x; i < a.zero_n; i += blockDim.x) a.zero[i] = 0;
  if (a.adv_len != nullptr && blockIdx.x == 0) {
    for (int32_t b = threadIdx.x; b < a.adv_B; b += blockDim.x)
      a.adv_len[b] = min(a.adv_len[b] + a.adv_T, a.adv_cap);
  }
  const int32_t chunks = a.head_dim / 16;
  const int64_t total = a.n_ids * chunks;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / chunks;
    const int32_t c = static_cast<int32_t>(i % chunks);
    const int32_t id = __ldg(a.ids + r);
    uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
    if (id >= 0 && id < a.num_rows) {
      const uint4 codes = __ldg(reinterpret_cast<const uint4*>(
          a.table + static_cast<int64_t>(id) * a.head_dim + c * 16));
      const uint32_t sc = __ldg(a.scales + static_cast<int64_t>(id) * (a.head_dim / 32) + c / 2);
      dequant16(codes, e8m0_to_f32(sc), lo, hi);
    } else {
      set_error(a.err, kErrIdRange);
    }
    uint4* dst = reinterpret_cast<uint4*>(a.out + r * a.head_dim + c * 16);
    dst[0] = lo;
    dst[1] = hi;
  }
}

// Stages 1 + 2 in one kernel, so the ids never make a round trip through memory, for one or
// several Engram layers (each with its own hash constants and table: Engram listing, __init__,
// layer_hash_index). A block takes `positions` consecutive positions: first one thread per
// (position, look-back k) resolves the compressed id c_{p-k} (token map, cache or pad) into
// shared memory once for all layers and appends c_p to the cache; then one thread per
// (position, layer, slot) forms the slot's mix and id from shared memory and gathers +
// dequantises its table row (independent 16-byte loads). `positions` is chosen so that a block's
// (position, layer, slot) items fit its threads, so all of their row loads are in flight at once.
constexpr int kHrMaxPositions = 8;
constexpr int kHrMaxNgram = 8;
constexpr int kHrThreads = 256;

__host__ __device__ inline int32_t hash_rows_positions(int32_t items_per_position) {
  const int32_t p = kHrThreads / items_per_position;
  return p < 1 ? 1 : (p > kHrMaxPositions ? kHrMaxPositions : p);
}

__global__ void __launch_bounds__(kHrThreads)
    hash_rows_kernel(const __grid_constant__ HashRowsArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  // the next kernel's counters (it reads them only after this grid has completed)
  if (a.zero != nullptr && blockIdx.x == 0)
    for (int32_t i = threadIdx.x; i < a.zero_n; i += blockDim.x) a.zero[i] = 0;
  const HashArgs& h = a.hash;
  const int32_t S = (h.max_ngram - 1) * h.n_heads;
  const int32_t LS = a.n_layers * S;   // items per position
  const int32_t P = a.positions;
  const int64_t M = static_cast<int64_t>(h.B) * h.T;
  const int64_t pos0 = static_cast<int64_t>(blockIdx.x) * P;
  __shared__ int32_t cwin[kHrMaxPositions][kHrMaxNgram];

  // The constants of this thread's first item (its layer's multipliers, its slot's prime and
  // offset) are fetched now, so that their loads overlap phase 1's instead of adding a round trip
  // to memory after it.
  const int32_t r_first = static_cast<int32_t>(threadIdx.x) % LS;
  const HashLayer& lf = a.layer[r_first / S];
  uint64_t mult[kHrMaxNgram];
#pragma unroll
  for (int k = 0; k < kHrMaxNgram; ++k) mult[k] = k < h.max_ngram ? __ldg(lf.multipliers + k) : 0;
  const uint64_t prime_first = __ldg(lf.primes + r_first % S);
  const int64_t offset_first = __ldg(lf.offsets + r_first % S);

  // phase 1: the window c_{p-k} of every position of the block
  if (threadIdx.x < P * h.max_ngram) {
    const int j = threadIdx.x / h.max_ngram, k = threadIdx.x % h.max_ngram;
    const int64_t bt = pos0 + j;
    if (bt < M) {
      const int32_t b = static_cast<int32_t>(bt / h.T), t = static_cast<int32_t>(bt % h.T);
      const int32_t len0 = h.cache_len[b];
      const int32_t c = compressed_id(h, b, t, len0, k);
      cwin[j][k] = c;
      if (k == 0) {
        const int64_t p = static_cast<int64_t>(len0) + t;
        if (p < h.capacity)
          h.cache[static_cast<int64_t>(b) * h.capacity + p] = c;
        else
          set_error(h.err, kErrCacheCapacity);
      }
    }
  }
  __syncthreads();

  // phase 2: slot ids and rows, item = (position j, layer l, slot s)
  const int32_t chunks = a.head_dim / 16;
  for (int item = threadIdx.x; item < P * LS; item += kHrThreads) {
    const int j = item / LS, r = item % LS;
    const int l = r / S, s = r % S;
    const int64_t bt = pos0 + j;
    if (bt >= M) break;
    const HashLayer& L = a.layer[l];
    const bool first = item == static_cast<int>(threadIdx.x);
    const int32_t n = s / h.n_heads + 2;
    uint64_t mix = 0;
#pragma unroll
    for (int32_t k = 0; k < kHrMaxNgram; ++k)
      if (k < n)
        mix ^= static_cast<uint64_t>(static_cast<int64_t>(cwin[j][k])) *
               (first ? mult[k] : __ldg(L.multipliers + k));
    const uint64_t prime = first ? prime_first : __ldg(L.primes + s);
    const int64_t offset = first ? offset_first : __ldg(L.offsets + s);
    const int32_t id = static_cast<int32_t>(static_cast<int64_t>(mix % prime) + offset);
    const int64_t i = bt * S + s;
    if (L.hash_ids) L.hash_ids[i] = id;
    uint4* dst = reinterpret_cast<uint4*>(L.rows + i * a.head_dim);
    if (id < 0 || id >= L.num_rows) {
      set_error(h.err, kErrIdRange);
      for (int32_t c = 0; c < 2 * chunks; ++c) dst[c] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* src =
        reinterpret_cast<const uint4*>(L.table + static_cast<int64_t>(id) * a.head_dim);
    const uint8_t* sc = L.scales + static_cast<int64_t>(id) * (a.head_dim / 32);
    const uint64_t once = l2_evict_first_policy();
    if (chunks == 4) {   // head_dim 64: all four loads in flight at once
      uint4 code[4];
      uint32_t scl[2];
#pragma unroll
      for (int c = 0; c < 4; ++c) code[c] = ldg_hint(src + c, once);
      scl[0] = ldg_u8_hint(sc, once);
      scl[1] = ldg_u8_hint(sc + 1, once);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 lo, hi;
        dequant16(code[c], e8m0_to_f32(scl[c / 2]), lo, hi);
        dst[2 * c] = lo;
        dst[2 * c + 1] = hi;
      }
    } else {
      for (int32_t c = 0; c < chunks; ++c) {
        uint4 lo, hi;
        dequant16(ldg_hint(src + c, once), e8m0_to_f32(ldg_u8_hint(sc + c / 2, once)), lo, hi);
        dst[2 * c] = lo;
        dst[2 * c + 1] = hi;
      }
    }
  }
}

HashRowsArgs single_layer_hash_rows(const HashArgs& h, const uint8_t* table,
                                    const uint8_t* scales, int64_t num_rows, int32_t head_dim,
                                    uint16_t* rows) {
  HashRowsArgs a{};
  a.hash = h;
  a.n_layers = 1;
  a.head_dim = head_dim;
  a.layer[0] = HashLayer{h.multipliers, h.primes, h.offsets, table, scales, num_rows, rows,
                         h.hash_ids};
  return a;
}

cudaError_t launch_hash_rows(const HashRowsArgs& args, cudaStream_t st, bool pdl) {
  if (args.hash.max_ngram > kHrMaxNgram || args.n_layers < 1 || args.n_layers > kMaxHashLayers)
    return cudaErrorInvalidValue;
  HashRowsArgs a = args;
  const int32_t S = (a.hash.max_ngram - 1) * a.hash.n_heads;
  const int64_t M = static_cast<int64_t>(a.hash.B) * a.hash.T;
  // As many positions per block as fit its threads, but no more than it takes to spread the
  // positions over every SM: with few positions (decode) each SM then has few row loads in
  // flight, which are latency-bound (a random 64-byte row of a large table each).
  int64_t P = hash_rows_positions(a.n_layers * S);
  const int64_t sms = device_sm_count();
  const int64_t spread = (M + sms - 1) / sms;
  if (spread < P) P = spread < 1 ? 1 : spread;
  a.positions = static_cast<int32_t>(P);
  const int64_t blocks = (M + P - 1) / P;
  return launch_ex(hash_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kHrThreads), 0, st,
                   pdl, a);
}

cudaError_t launch_rows(const RowsArgs& a, cudaStream_t st, bool pdl) {
  const int64_t total = a.n_ids * (a.head_dim / 16);
  int64_t blocks = (total + 255) / 256;
  if (blocks < 1) blocks = 1;
  if (blocks > (1 << 20)) blocks = 1 << 20;
  return launch_ex(rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, pdl, a);
}

// -------------------------------------------------------------------- stage 4: gate and add
// Engram listing, forward after the projection; page "DeepSeek V4.1 · Gate per stream".
// One block per (token, stream): reduce sum h^2, sum key^2, sum h*w*key over dim (16-byte loads,
// warp shuffles), form the gate, then write h + gate * value (x re-read from L1/L2).

constexpr int kGateThreads = 256;

// 8 consecutive kv values (one 16-byte bf16 word) at column n of token m: either read from the
// bf16 kv, or the f32 partial sums of the split-K projection added in K order and rounded once.
__device__ __forceinline__ uint4 load_kv8(const GateArgs& a, int64_t m, int64_t N, int64_t n) {
  if (a.part == nullptr) return __ldg(reinterpret_cast<const uint4*>(a.kv + m * N + n));
  float v[8];
  const float4* p0 = reinterpret_cast<const float4*>(a.part + m * N + n);
  float4 lo = __ldg(p0), hi = __ldg(p0 + 1);
  v[0] = lo.x; v[1] = lo.y; v[2] = lo.z; v[3] = lo.w;
  v[4] = hi.x; v[5] = hi.y; v[6] = hi.z; v[7] = hi.w;
  for (int k = 1; k < a.ksplit; ++k) {
    const float4* pk = reinterpret_cast<const float4*>(a.part + (k * a.M + m) * N + n);
    lo = __ldg(pk);
    hi = __ldg(pk + 1);
    v[0] += lo.x; v[1] += lo.y; v[2] += lo.z; v[3] += lo.w;
    v[4] += hi.x; v[5] += hi.y; v[6] += hi.z; v[7] += hi.w;
  }
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}

__device__ __forceinline__ void advance_lengths(const LenAdvance& adv) {
  if (adv.len != nullptr && blockIdx.x == 0)
    for (int32_t b = threadIdx.x; b < adv.B; b += blockDim.x)
      adv.len[b] = min(adv.len[b] + adv.T, adv.cap);
}

__device__ __forceinline__ void acc_sums(uint4 xv, uint4 kv, uint4 qv, uint4 wv, float& sh2,
                                         float& sk2, float& shwk) {
  const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w}, ks[4] = {kv.x, kv.y, kv.z, kv.w};
  const uint32_t qs[4] = {qv.x, qv.y, qv.z, qv.w}, ws[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int sh = half * 16;
      const float h = bf16_bits_to_f32((xs[j] >> sh) & 0xFFFFu);
      const float kk = bf16_bits_to_f32((ks[j] >> sh) & 0xFFFFu);
      const float w = bf16_bits_to_f32((qs[j] >> sh) & 0xFFFFu) *
                      bf16_bits_to_f32((ws[j] >> sh) & 0xFFFFu);
      sh2 = fmaf(h, h, sh2);
      sk2 = fmaf(kk, kk, sk2);
      shwk = fmaf(h * w, kk, shwk);
    }
  }
}

__device__ __forceinline__ uint4 gate_out8(uint4 xv, uint4 vv, float g) {
  const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w}, vs[4] = {vv.x, vv.y, vv.z, vv.w};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float h0 = bf16_bits_to_f32(xs[j] & 0xFFFFu), h1 = bf16_bits_to_f32(xs[j] >> 16);
    const float v0 = bf16_bits_to_f32(vs[j] & 0xFFFFu), v1 = bf16_bits_to_f32(vs[j] >> 16);
    o[j] = pack_bf16x2(fmaf(g, v0, h0), fmaf(g, v1, h1));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Block reduction of the three sums; returns the gate (0 for a masked token) to every thread.
__device__ __forceinline__ float block_gate(const GateArgs& a, int64_t m, int32_t s, float sh2,
                                            float sk2, float shwk) {
  __shared__ float red[3][kGateThreads / 32];
  __shared__ float gate_s;
  sh2 = warp_sum(sh2);
  sk2 = warp_sum(sk2);
  shwk = warp_sum(shwk);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red[0][warp] = sh2;
    red[1][warp] = sk2;
    red[2][warp] = shwk;
  }
  __syncthreads();
  if (warp == 0) {
    float r0 = lane < kGateThreads / 32 ? red[0][lane] : 0.f;
    float r1 = lane < kGateThreads / 32 ? red[1][lane] : 0.f;
    float r2 = lane < kGateThreads / 32 ? red[2][lane] : 0.f;
    r0 = warp_sum(r0);
    r1 = warp_sum(r1);
    r2 = warp_sum(r2);
    if (lane == 0) {
      const bool keep = a.mask == nullptr || a.mask[m] != 0;
      const float g = keep ? gate_from_sums(r0, r1, r2, a.dim, a.eps, a.inv_sqrt_dim) : 0.f;
      gate_s = g;
      if (a.gate_out) a.gate_out[m * a.hc + s] = g;
    }
  }
  __syncthreads();
  return gate_s;
}

// One block per (token, stream). kVec > 0: each thread keeps its (at most kVec) 8-element
// vectors of x, key and value in registers (dim <= 8 * kVec * kGateThreads), and the value loads
// are issued before the reduction; kVec == 0: any dim, two passes over x.
template <int kVec>
__global__ void __launch_bounds__(kGateThreads) gate_kernel(GateArgs a) {
  const int64_t m = blockIdx.x / a.hc;
  const int32_t s = blockIdx.x % a.hc;
  const int64_t N = static_cast<int64_t>(a.dim) * (a.hc + 1);
  const uint16_t* xr = a.x + (m * a.hc + s) * a.dim;
  const int64_t key0 = static_cast<int64_t>(s) * a.dim;      // first key column of stream s
  const int64_t val0 = static_cast<int64_t>(a.hc) * a.dim;   // first value column
  const uint16_t* qr = a.q + static_cast<int64_t>(s) * a.dim;
  const uint16_t* kr = a.k + static_cast<int64_t>(s) * a.dim;
  const int nvec = a.dim / 8;
  const bool keep = a.mask == nullptr || a.mask[m] != 0;
  const bool write_value = a.kv_out != nullptr && s == 0;
  uint16_t* orow = a.out + (m * a.hc + s) * a.dim;
  float sh2 = 0.f, sk2 = 0.f, shwk = 0.f;

  if constexpr (kVec > 0) {
    // x, q, k and the mask are inputs of the forward that no kernel of its chain writes: they are
    // loaded before waiting for the projection (the kernel ahead of this one in the stream)
    uint4 xv[kVec], qv[kVec], kw[kVec], vv[kVec];
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
      const int v = threadIdx.x + j * kGateThreads;
      if (v < nvec) {
        xv[j] = __ldg(reinterpret_cast<const uint4*>(xr) + v);
        qv[j] = __ldg(reinterpret_cast<const uint4*>(qr) + v);
        kw[j] = __ldg(reinterpret_cast<const uint4*>(kr) + v);
      }
    }
    pdl_wait();
    pdl_launch_dependents();
    advance_lengths(a.adv);
    // every key and value load is issued before the first is used: the warp issues in order,
    // so a use between them would wait out each load's latency in turn
    uint4 kvk[kVec];
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
      const int v = threadIdx.x + j * kGateThreads;
      if (v < nvec) {
        kvk[j] = load_kv8(a, m, N, key0 + 8 * v);
        if (keep || write_value) vv[j] = load_kv8(a, m, N, val0 + 8 * v);
      }
    }
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
      const int v = threadIdx.x + j * kGateThreads;
      if (v < nvec) {
        if (a.kv_out) reinterpret_cast<uint4*>(a.kv_out + m * N + key0)[v] = kvk[j];
        acc_sums(xv[j], kvk[j], qv[j], kw[j], sh2, sk2, shwk);
      }
    }
    const float g = block_gate(a, m, s, sh2, sk2, shwk);
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
      const int v = threadIdx.x + j * kGateThreads;
      if (v < nvec) {
        if (write_value) reinterpret_cast<uint4*>(a.kv_out + m * N + val0)[v] = vv[j];
        // a masked token's x passes through unchanged
        reinterpret_cast<uint4*>(orow)[v] = keep ? gate_out8(xv[j], vv[j], g) : xv[j];
      }
    }
  } else {
    pdl_wait();
    pdl_launch_dependents();
    advance_lengths(a.adv);
    for (int v = threadIdx.x; v < nvec; v += kGateThreads) {
      const uint4 kv = load_kv8(a, m, N, key0 + 8 * v);
      if (a.kv_out) reinterpret_cast<uint4*>(a.kv_out + m * N + key0)[v] = kv;
      acc_sums(__ldg(reinterpret_cast<const uint4*>(xr) + v), kv,
               __ldg(reinterpret_cast<const uint4*>(qr) + v),
               __ldg(reinterpret_cast<const uint4*>(kr) + v), sh2, sk2, shwk);
    }
    const float g = block_gate(a, m, s, sh2, sk2, shwk);
    for (int v = threadIdx.x; v < nvec; v += kGateThreads) {
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(xr) + v);
      if (!keep && !write_value) {
        reinterpret_cast<uint4*>(orow)[v] = xv;
        continue;
      }
      const uint4 vv = load_kv8(a, m, N, val0 + 8 * v);
      if (write_value) reinterpret_cast<uint4*>(a.kv_out + m * N + val0)[v] = vv;
      reinterpret_cast<uint4*>(orow)[v] = keep ? gate_out8(xv, vv, g) : xv;
    }
  }
}

// out = h + gate * value for (token m, stream s) from the fused kernel's deferred output: its gates
// and bf16 value rows. x and the mask are inputs no kernel of the forward writes, so they are
// loaded before waiting for the fused kernel.
template <int kVec>
__global__ void __launch_bounds__(kGateThreads) gate_apply_kernel(GateApplyArgs a) {
  const int64_t m = blockIdx.x / a.hc;
  const int32_t s = blockIdx.x % a.hc;
  const uint16_t* xr = a.x + (m * a.hc + s) * a.dim;
  const int nvec = a.dim / 8;
  const bool keep = a.mask == nullptr || a.mask[m] != 0;
  uint16_t* orow = a.out + (m * a.hc + s) * a.dim;
  uint4 xv[kVec], vv[kVec];
#pragma unroll
  for (int j = 0; j < kVec; ++j) {
    const int v = threadIdx.x + j * kGateThreads;
    if (v < nvec) xv[j] = __ldg(reinterpret_cast<const uint4*>(xr) + v);
  }
  pdl_wait();
  pdl_launch_dependents();
  const float g = keep ? a.gx[m * a.hc + s] : 0.f;
#pragma unroll
  for (int j = 0; j < kVec; ++j) {
    const int v = threadIdx.x + j * kGateThreads;
    if (v < nvec && keep) vv[j] = __ldg(reinterpret_cast<const uint4*>(a.value + m * a.dim) + v);
  }
#pragma unroll
  for (int j = 0; j < kVec; ++j) {
    const int v = threadIdx.x + j * kGateThreads;
    if (v < nvec)   // a masked token's x passes through unchanged
      reinterpret_cast<uint4*>(orow)[v] = keep ? gate_out8(xv[j], vv[j], g) : xv[j];
  }
}

cudaError_t launch_gate_apply(const GateApplyArgs& a, cudaStream_t st, bool pdl) {
  const dim3 grid(static_cast<unsigned>(a.M * a.hc)), block(kGateThreads);
  const int nvec = a.dim / 8;
  if (nvec <= 1 * kGateThreads) return launch_ex(gate_apply_kernel<1>, grid, block, 0, st, pdl, a);
  if (nvec <= 2 * kGateThreads) return launch_ex(gate_apply_kernel<2>, grid, block, 0, st, pdl, a);
  if (nvec <= 3 * kGateThreads) return launch_ex(gate_apply_kernel<3>, grid, block, 0, st, pdl, a);
  if (nvec <= 4 * kGateThreads) return launch_ex(gate_apply_kernel<4>, grid, block, 0, st, pdl, a);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gate(const GateArgs& a, cudaStream_t st, bool pdl) {
  const dim3 grid(static_cast<unsigned>(a.M * a.hc)), block(kGateThreads);
  const int nvec = a.dim / 8;
  if (nvec <= 1 * kGateThreads) return launch_ex(gate_kernel<1>, grid, block, 0, st, pdl, a);
  if (nvec <= 2 * kGateThreads) return launch_ex(gate_kernel<2>, grid, block, 0, st, pdl, a);
  if (nvec <= 3 * kGateThreads) return launch_ex(gate_kernel<3>, grid, block, 0, st, pdl, a);
  if (nvec <= 4 * kGateThreads) return launch_ex(gate_kernel<4>, grid, block, 0, st, pdl, a);
  return launch_ex(gate_kernel<0>, grid, block, 0, st, pdl, a);
}

}  // namespace engram
