// The decode step's stages 1-3 in one kernel, for up to 64 tokens: every CTA hashes the batch's
// positions and gathers their table rows itself, while its share of the wkv weight is already
// streaming into shared memory, then projects, and leaves for the gate only the value rows and
// per-32-column partial sums of the keys.
//
// Page "Module engram", stages 1-3 (NgramHashState; embed_rows; linear_bf16) and the Engram
// listing's forward up to the split of kv into keys and value.
//
// Why every CTA hashes: a decode step is bound by streaming the 78.6 MB weight once. A separate
// hash-and-gather kernel in front of the projection is a chain of dependent cold loads (cache
// length, window, token map, table row) plus a grid-wide completion before the projection may
// read its activation; the weight stream waits behind it. Here the weight's first stages are
// requested at the kernel's start and the activation is produced inside the CTA, so the only
// dependency the stream meets is the CTA's own gather (three dependent loads). The repeated
// hashing costs L2 traffic (each CTA reads the same 64 x 24 rows, ~100 KB) and ALU time that the
// weight stream hides.
//
// Weight layout on the SMs: units of 64 wkv rows (400 at full width); CTA i owns units i,
// i + grid, i + 2 * grid (at most three). A ring stage holds one 64-row weight box per unit
// (TMA) and the activation box of one K-block (64 tokens x 64 K, written by the gather threads in
// the 128-byte swizzle a TMA load would produce). Two units share one tcgen05 MMA (kind::f16,
// M = 128, N = tokens rounded up to 32); a third unit's MMA has whatever the next box holds in
// rows 64-127, whose products are never read.
//
// Epilogue, per kv column (one TMEM lane) and token: kv = bf16(acc). Key columns contribute
// sum key^2 and sum h * w * key over their 32-column group (w = q * k), reduced across the warp
// in a fixed order and stored per (group, token); value columns are stored as bf16 rows. The gate
// kernel that follows adds the 32-column partial sums of a (token, stream) in group order.
//
// Roles (320 threads): warp 0 TMA producer; warp 1 TMEM owner and MMA issuer; warps 2-9 hash,
// gather and write the activation boxes, then run the epilogue.
#include "device.cuh"
#include "hash_rows.cuh"
#include "decode_step.h"
#include "kernels.h"
#include "wkv_tiles.cuh"

namespace engram {

namespace {

constexpr int kDsThreads = 320;
constexpr int kDsGather = 256;                   // gather / epilogue threads (warps 2-9)
constexpr int kDsRows = 64;                      // wkv rows per unit
constexpr int kDsMaxTokens = 64;
constexpr int kDsMaxUnits = 3;
constexpr int kDsBoxBytes = kDsRows * kBK * 2;   // 8 KB
constexpr int kDsStageBytes = (kDsMaxUnits + 1) * kDsBoxBytes;
constexpr int kDsStages = 6;
constexpr int kDsSlotClasses = 4;                // thread g hashes slots g / 64 + 4 j
constexpr int kDsMaxSlotsPerThread = 6;          // up to 24 hash columns
constexpr int kDsMaxNgram = 4;                   // look-backs k = cls (one per slot class)
constexpr int kDsMaxSlots = kDsSlotClasses * kDsMaxSlotsPerThread;
constexpr uint32_t kDsTmemCols = 128;            // two accumulators (unit pairs) of <= 64 columns
constexpr int kDsXBoxBytes = kDsMaxTokens * kDsRows * 2;   // x of one unit's 64 columns: 8 KB

struct DsShared {
  uint64_t full[kDsStages];
  uint64_t empty[kDsStages];
  uint64_t tfull;
  uint64_t drain;
  uint64_t go;      // the weight stream may start (the hash window has been read)
  uint64_t xfull;   // the x boxes of the CTA's key units have landed
  uint32_t tmem_base;
  int abort;
  int32_t cwin[kDsMaxTokens][kDsMaxNgram];
  int32_t ids[kDsMaxTokens][kDsMaxSlots];
  uint64_t prime[kDsMaxSlots];
  uint64_t magic[kDsMaxSlots];   // mod_magic_u64(prime)
};

size_t ds_smem_bytes() {
  return size_t(kDsStages) * kDsStageBytes + size_t(kDsMaxUnits) * kDsXBoxBytes +
         sizeof(DsShared) + 1024;
}

// Transpose-reduce of 32 values per lane across the warp: afterwards v[0] of lane j holds the sum
// over all lanes of their v[j]. Fixed order (a butterfly), so results do not vary run to run.
__device__ __forceinline__ void warp_transpose_sum(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? v[i] : v[i + o];
      const float keep = upper ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
    }
  }
}

// Issue the loads of slot `slot`'s rows for thread (tq, c4) of a slot class: chunk c4 of the rows
// of positions tq + 16 i (zero beyond the batch, or for an id outside the table, which also sets
// the error bit), and the scale pair of position tq + 16 c4 (0x7F7F, unit scales, where there is
// no row). The loads are pinned, so their results stay in registers until used.
__device__ __forceinline__ void ds_issue_rows(const DecodeStepArgs& a, const DsShared* sh,
                                              int slot, int tq, int c4, uint4 (&r)[4],
                                              uint32_t& scale_pair) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    r[i] = make_uint4(0, 0, 0, 0);
    const int pos = tq + 16 * i;
    if (pos >= a.M) continue;
    const int32_t id = sh->ids[pos][slot];
    if (id < 0 || id >= a.num_rows) {
      if (c4 == 0) set_error(a.err, kErrIdRange);
      continue;
    }
    r[i] = ldg_pinned_v4(a.table + static_cast<int64_t>(id) * 64 + c4 * 16);
  }
  scale_pair = 0x7F7Fu;
  const int pos = tq + 16 * c4;
  if (pos < a.M) {
    const int32_t id = sh->ids[pos][slot];
    if (id >= 0 && id < a.num_rows)
      scale_pair = ldg_pinned_u16(a.scales + static_cast<int64_t>(id) * 2);
  }
}

__global__ void __launch_bounds__(kDsThreads, 1)
    engram_decode_kernel(const __grid_constant__ CUtensorMap tmW,
                         const __grid_constant__ CUtensorMap tmX,
                         const __grid_constant__ DecodeStepArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint8_t* xbox = smem + kDsStages * kDsStageBytes;   // x of unit i at xbox + i * 8 KB
  DsShared* sh = reinterpret_cast<DsShared*>(xbox + kDsMaxUnits * kDsXBoxBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kblocks = a.K / kBK;
  const int32_t units_total = a.N / kDsRows;
  int32_t units[kDsMaxUnits];
  int nu = 0;
  for (int32_t u = blockIdx.x; u < units_total && nu < kDsMaxUnits; u += gridDim.x)
    units[nu++] = u;
  const int npairs = (nu + 1) / 2;
  const uint32_t tok_off = static_cast<uint32_t>(kDsMaxUnits) * kDsBoxBytes;
  const uint32_t stage_tx = static_cast<uint32_t>(nu) * kDsBoxBytes;
  const int64_t key_cols = static_cast<int64_t>(a.hc) * a.dim;
  int nkey = 0;   // units whose columns are keys (the epilogue needs their x)
  for (int i = 0; i < nu; ++i) nkey += static_cast<int64_t>(units[i]) * kDsRows < key_cols;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kDsStages; ++i) {
      mbar_init(&sh->full[i], 3);   // the producer's expect_tx + the two warps writing the box
      mbar_init(&sh->empty[i], 1);
    }
    mbar_init(&sh->tfull, 1);
    mbar_init(&sh->drain, 1);
    mbar_init(&sh->go, 1);
    mbar_init(&sh->xfull, 1);
    sh->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(&sh->tmem_base, kDsTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;
  volatile int* abort = &sh->abort;
  // Every input may have been written by the kernel ahead of this one in the stream; nothing is
  // read before it has completed. The gate kernel after this one may start launching now.
  pdl_wait();
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------- TMA producer (weight only)
    if (lane == 0 && nu > 0) {
      // The weight's first stages are requested once the hash window has been read: its cold
      // loads are the head of the dependent chain to the activation, and queued behind a
      // 20 MB burst they take twice as long.
      TmaRingT<kDsStages> ring;
      const bool go = mbar_wait(&sh->go, 0, abort, a.err);
      for (int kb = 0; kb < kblocks && go; ++kb) {
        if (kb >= kDsStages && !ring.acquire(sh->empty, abort, a.err)) break;
        uint8_t* st = smem + ring.stage * kDsStageBytes;
        mbar_arrive_expect_tx(&sh->full[ring.stage], stage_tx);
        for (int i = 0; i < nu; ++i)
          tma_load_2d(st + i * kDsBoxBytes, &tmW, &sh->full[ring.stage], kb * kBK,
                      units[i] * kDsRows);
        ring.issued();
        if (kb + 1 == (kblocks < kDsStages ? kblocks : kDsStages) && nkey > 0) {
          // after the first stages: x of the key units (tokens beyond M read as zero)
          mbar_arrive_expect_tx(&sh->xfull, static_cast<uint32_t>(nkey) * kDsXBoxBytes);
          for (int i = 0; i < nu; ++i) {
            const int64_t n0 = static_cast<int64_t>(units[i]) * kDsRows;
            if (n0 < key_cols)
              tma_load_3d(xbox + i * kDsXBoxBytes, &tmX, &sh->xfull,
                          static_cast<int32_t>(n0 % a.dim), static_cast<int32_t>(n0 / a.dim), 0);
          }
        }
      }
      ring.drain(sh->full);
      if (go && nkey > 0) mbar_wait_drain(&sh->xfull, 0);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0 && nu > 0) {
      const uint32_t idesc = idesc_bf16_f32(128, a.nt);
      uint32_t st = 0, ph = 0;
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait(&sh->full[st], ph, abort, a.err)) { ok = false; break; }
        tc_fence_after();
        const uint8_t* sp = smem + st * kDsStageBytes;
        const uint64_t bd = sw128_kmajor_desc(smem_u32(sp + tok_off));
        for (int pr = 0; pr < npairs; ++pr) {
          const uint64_t ad = sw128_kmajor_desc(smem_u32(sp + 2 * pr * kDsBoxBytes));
          const uint32_t d = tmem_base + pr * (kDsTmemCols / 2);
#pragma unroll
          for (int kk = 0; kk < kBK / kUmmaK; ++kk)
            tc_mma_bf16(d, ad + 2ull * kk, bd + 2ull * kk, idesc, (kb | kk) != 0);
        }
        tc_commit(&sh->empty[st]);
        if (++st == kDsStages) { st = 0; ph ^= 1u; }
      }
      if (ok) tc_commit(&sh->tfull);
      tc_commit(&sh->drain);
      mbar_wait_drain(&sh->drain, 0);
    }
  } else {
    // ------------------------------------------------- hash + gather (warps 2-9), then epilogue
    const int g = threadIdx.x - 64;
    const HashArgs& h = a.hash;
    const int S = (h.max_ngram - 1) * h.n_heads;
    {
      // the ids: thread (q, cls) forms those of slots cls, cls + 4, ... of position q
      const int q = g & (kDsMaxTokens - 1), cls = g >> 6;
      const int js = S / kDsSlotClasses;
      const bool live = q < a.M;
      if (a.ids != nullptr) {   // given (the listing's forward(x, hash_ids, token_mask))
        if (g == 0) mbar_arrive(&sh->go);
        for (int j = 0; j < js; ++j)
          sh->ids[q][cls + 4 * j] =
              live ? __ldg(a.ids + static_cast<int64_t>(q) * S + cls + 4 * j) : 0;
      } else {
        // the slots' reciprocals for the modulo, one slot per thread, formed while the window
        // loads are in flight; the multipliers and offsets of this thread's slots likewise
        if (g < S) {
          const uint64_t P = __ldg(h.primes + g);
          sh->prime[g] = P;
          sh->magic[g] = mod_magic_u64(P);
        }
        uint64_t mult[kDsMaxNgram];
        int64_t off[kDsMaxSlotsPerThread];
#pragma unroll
        for (int k = 0; k < kDsMaxNgram; ++k)
          mult[k] = k < h.max_ngram ? __ldg(h.multipliers + k) : 0;
#pragma unroll
        for (int j = 0; j < kDsMaxSlotsPerThread; ++j)
          off[j] = j < js ? __ldg(h.offsets + cls + 4 * j) : 0;
        // the window c_{q-k}: thread (q, cls) resolves look-back k = cls
        if (live && cls < h.max_ngram) {
          const int32_t b = q / h.T, t = q % h.T;
          const int32_t len0 = h.cache_len[b];
          const int32_t c = compressed_id(h, b, t, len0, cls);
          sh->cwin[q][cls] = c;
          if (cls == 0 && blockIdx.x == 0) {   // one CTA appends c_q to the cache
            const int64_t pos = static_cast<int64_t>(len0) + t;
            if (pos < h.capacity)
              h.cache[static_cast<int64_t>(b) * h.capacity + pos] = c;
            else
              set_error(h.err, kErrCacheCapacity);
          }
        }
        named_bar_sync(1, kDsGather);
        if (g == 0) mbar_arrive(&sh->go);
#pragma unroll
        for (int j = 0; j < kDsMaxSlotsPerThread; ++j) {
          if (j >= js) break;
          const int s = cls + 4 * j;
          int32_t id = 0;
          if (live) {
            const int n = s / h.n_heads + 2;
            uint64_t mix = 0;
#pragma unroll
            for (int k = 0; k < kDsMaxNgram; ++k)
              if (k < n)
                mix ^= static_cast<uint64_t>(static_cast<int64_t>(sh->cwin[q][k])) * mult[k];
            id = static_cast<int32_t>(
                static_cast<int64_t>(mod_u64_by(mix, sh->prime[s], sh->magic[s])) + off[j]);
            if (blockIdx.x == 0 && h.hash_ids != nullptr)
              h.hash_ids[static_cast<int64_t>(q) * S + s] = id;
          }
          sh->ids[q][s] = id;
        }
      }
      named_bar_sync(1, kDsGather);
    }

    // the rows: the 64 threads of slot class cls (warps 2 + 2 cls and 3 + 2 cls) gather the rows
    // of slots cls + 4 j and write them, dequantised, as the activation boxes of K-blocks
    // cls + 4 j. Thread (tq, c4) of the class holds 16-byte chunk c4 of the rows of positions
    // tq + 16 i, i = 0..3: the four threads of a row are adjacent lanes, so each row is one
    // 64-byte request (152 CTAs read the same 64 x 24 rows). The rows of two slots are in flight
    // ahead of the box being written, so K-block 0 waits for one slot's rows, not for all of them.
    const int cls = g >> 6, tq = (g & 63) >> 2, c4 = g & 3;
    const int js = S / kDsSlotClasses;
    uint4 cur[4], nxt[4];
    uint32_t scur = 0, snxt = 0;
    if (js > 0) ds_issue_rows(a, sh, cls, tq, c4, cur, scur);
    if (js > 1) ds_issue_rows(a, sh, cls + 4, tq, c4, nxt, snxt);

    // The loop is kept rolled, with one copy of the dequantisation: eight warps run it at
    // different K-blocks, and an unrolled copy per K-block would not stay in the instruction
    // cache.
    bool ok = true;
#pragma unroll 1
    for (int j = 0; j < js; ++j) {
      const int kb = cls + 4 * j;
      const int st = kb % kDsStages, round = kb / kDsStages;
      if (round > 0) {
        bool w = mbar_wait(&sh->empty[st], static_cast<uint32_t>(round - 1) & 1u, abort, a.err);
        ok = __all_sync(0xFFFFFFFFu, w);
        if (!ok) break;
      }
      const uint32_t box = smem_u32(smem + st * kDsStageBytes + tok_off);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // the scale pair of position tq + 16 i was loaded by lane c4 = i of the row's group
        const uint32_t pair = __shfl_sync(0xFFFFFFFFu, scur, (lane & ~3) | i);
        const int pos = tq + 16 * i;
        if (pos >= a.nt) continue;
        uint4 lo, hi;
        dequant16(cur[i], e8m0_to_f32((pair >> (8 * (c4 >> 1))) & 0xFFu), lo, hi);
        const uint32_t rbase = box + pos * 128;
        sts128(rbase + ((static_cast<uint32_t>(2 * c4) ^ (pos & 7)) << 4), lo);
        sts128(rbase + ((static_cast<uint32_t>(2 * c4 + 1) ^ (pos & 7)) << 4), hi);
      }
      fence_proxy_async_shared();   // the tensor core reads the box through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->full[st]);
#pragma unroll
      for (int i = 0; i < 4; ++i) cur[i] = nxt[i];
      scur = snxt;
      if (j + 2 < js) ds_issue_rows(a, sh, cls + 4 * (j + 2), tq, c4, nxt, snxt);
    }

    // ------------------------------------------------------------- epilogue
    const int quad = warp & 3;               // TMEM lane quadrant this warp may read
    const int half = (warp - 2) >> 2;        // tokens 32 * half .. + 31
    const bool run = ok && nu > 0 && 32 * half < a.nt;
    // the w = q * k of this thread's key columns, requested before the last MMAs complete
    float wcol[2] = {0.f, 0.f};
    int64_t col[2] = {-1, -1};
    bool any_key = false;
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
      const int ui = 2 * pr + (quad >> 1);
      if (!run || pr >= npairs || ui >= nu) continue;
      const int64_t n = static_cast<int64_t>(units[ui]) * kDsRows + (quad & 1) * 32 + lane;
      col[pr] = n;
      if (n >= key_cols) continue;
      any_key = true;
      wcol[pr] = bf16_bits_to_f32(ldg_pinned_u16(a.q + n)) * bf16_bits_to_f32(ldg_pinned_u16(a.k + n));
    }
    bool ready = run && mbar_wait(&sh->tfull, 0, abort, a.err);
    if (ready && any_key) ready = mbar_wait(&sh->xfull, 0, abort, a.err);
    ready = __all_sync(0xFFFFFFFFu, ready);
    if (ready) {
      tc_fence_after();
#pragma unroll 1
      for (int pr = 0; pr < npairs; ++pr) {
        const int64_t n = pr == 0 ? col[0] : col[1];
        if (n < 0) continue;   // warp-uniform
        const float wp = pr == 0 ? wcol[0] : wcol[1];
        // x of this column for token m in the unit's x box (128-byte swizzled rows of 64 columns)
        const int cu = (quad & 1) * 32 + lane;
        const uint32_t xrow = smem_u32(xbox + (2 * pr + (quad >> 1)) * kDsXBoxBytes) + (cu & 7) * 2;
        uint32_t r[32];
        tc_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             pr * (kDsTmemCols / 2) + half * 32,
                         r);
        tc_wait_ld(r);
        // One path for key and value columns (the stores are predicated): the second pair then
        // runs instructions the first has already brought into the instruction cache.
        // (The key/value choice enters as data, a mask and a token limit, so that the compiler
        // has no branch to duplicate the loops under.)
        const bool is_key = n < key_cols;
        const uint32_t xmask = is_key ? 0xFFFFu : 0u;   // a value unit's x box holds no x
        const int vlim = is_key ? 0 : a.M;               // tokens whose value row is stored
        float kvb[32], k2[32], hwk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int m = 32 * half + i;
          kvb[i] = round_bf16(__uint_as_float(r[i]));
          const float hx = bf16_bits_to_f32(
              lds_u16(xrow + m * 128 + ((static_cast<uint32_t>(cu >> 3) ^ (m & 7)) << 4)) & xmask);
          k2[i] = kvb[i] * kvb[i];
          hwk[i] = (hx * wp) * kvb[i];
        }
        if (a.kv_out != nullptr) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int m = 32 * half + i;
            if (m < a.M)
              a.kv_out[static_cast<int64_t>(m) * a.N + n] =
                  static_cast<uint16_t>(pack_bf16x2(kvb[i], 0.f));
          }
        }
        warp_transpose_sum(k2, lane);
        warp_transpose_sum(hwk, lane);
        // key columns: the two sums of this warp's 32-column group for token 32 * half + lane
        if (is_key)
          a.part[(n >> 5) * kDsMaxTokens + 32 * half + lane] = make_float2(k2[0], hwk[0]);
        // value columns: the bf16 value rows
        const int64_t vc = is_key ? 0 : n - key_cols;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int m = 32 * half + i;
          if (m < vlim)
            a.value[static_cast<int64_t>(m) * a.dim + vc] =
                static_cast<uint16_t>(pack_bf16x2(kvb[i], 0.f));
        }
      }
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncwarp();
  cta_sync_all();   // every role is done with TMEM (each thread counted on its own)
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kDsTmemCols);
  }
}

}  // namespace

bool decode_step_supported(int64_t M, const DecodeGeometry& g) {
  const int S = (g.max_ngram - 1) * g.n_heads;
  const int32_t N = g.dim * (g.hc + 1);
  return M >= 1 && M <= kDsMaxTokens && g.head_dim == 64 && S % kDsSlotClasses == 0 &&
         S / kDsSlotClasses <= kDsMaxSlotsPerThread && g.max_ngram <= kDsMaxNgram &&
         S <= kDsGather &&
         g.dim % kDsRows == 0 && N / kDsRows <= kDsMaxUnits * device_sm_count();
}

size_t decode_step_part_bytes(int32_t hc, int32_t dim) {
  return size_t(hc) * dim / 32 * kDsMaxTokens * sizeof(float2);
}

cudaError_t launch_decode_step(const DecodeStepArgs& args, cudaStream_t st, bool pdl) {
  DecodeStepArgs a = args;
  a.nt = static_cast<int32_t>((a.M + 31) / 32 * 32);
  const int32_t units = a.N / kDsRows;
  const int32_t grid = units < device_sm_count() ? units : device_sm_count();
  alignas(64) CUtensorMap tmW, tmX;
  if (!tensor_map_2d_bf16(&tmW, a.w, a.K, a.N, kBK, kDsRows) ||
      !tensor_map_3d_bf16(&tmX, a.x, a.dim, a.hc, a.M, kDsRows, 1, kDsMaxTokens))
    return cudaErrorInvalidValue;
  const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(engram_decode_kernel),
                                            ds_smem_bytes());
  if (e != cudaSuccess) return e;
  return launch_ex(engram_decode_kernel, dim3(static_cast<unsigned>(grid)), dim3(kDsThreads),
                   ds_smem_bytes(), st, pdl, tmW, tmX, a);
}

}  // namespace engram
