// Stages 3 + 4 fused: the wkv projection on the tensor cores with the gate-and-add in its
// epilogue, so the dim * (hc + 1)-wide kv row never goes to HBM.
//
// Engram listing, forward: kv = wkv(rows); key, value = split(kv); per (token, stream) the three
// sums over dim (h^2, key^2, h*w*key) give the gate; out = bf16(h + gate * value).
//
// Work split. The kernel is persistent: as many CTA pairs (2-CTA clusters) as fit on the GPU at
// once, one CTA per SM. The work is cut into items of 256 tokens times one
// column tile of kv: a key tile (256 key columns of one stream) or a value tile (256 value
// columns, shared by every stream). Pairs take items from a global counter in the order of
// fused_schedule.cuh, so every SM stays busy to the end whatever the token count, and a pair that
// runs slow simply takes fewer items.
//
// Each item is a CTA-pair MMA (tcgen05 cta_group::2, M = 256): CTA h of the pair stages rows
// [128h, 128h + 128) of the 256 tokens and half of the tile's wkv rows per K-block, and gets its
// 128-row half of the accumulator in its own TMEM. The even CTA issues the MMAs; both CTAs' TMA
// loads count on its barriers and its commits arrive on the barriers of both.
//
// Key item epilogue: per token, the three sums over the tile's 256 columns, written to a partial
// buffer. The gate warp then counts the tile in (an atomic per token tile, half and stream); the
// CTA that completes the last key tile of (token tile, half, stream) adds the partial sums in
// column order (so the result does not depend on which pair ran what), forms the gates, and
// publishes them with a release flag. Value item epilogue: wait (bounded) for the flags of every
// stream of its tokens, then out[m, s, cols] = h + gate[m, s] * value for every stream s, computed
// in place in the x box in shared memory and written back with a TMA store.
//
// Roles per CTA (384 threads):
//   warp 0       TMA producer of this CTA's half of the GEMM operands, 5-stage ring; in the even
//                CTA it also takes the items from the global counter and hands them to both CTAs
//                through a small item ring in shared memory;
//   warp 1       TMEM owner; in the even CTA also the MMA issuer (two 256-column accumulators);
//   warps 2-9    epilogue: two warps per TMEM lane quadrant (warp w reads lanes 32*(w%4)...),
//                thread = (token row, half of each 64-column box): tcgen05.ld, gate sums, output;
//   warp 10      TMA producer of the residual streams x: 128-token x 64-column boxes into a
//                4-slot ring, in exactly the order the epilogue consumes them;
//   warp 11      gate warp: counts each key tile in and, for the last one, forms and publishes the
//                gates, off the epilogue's path.
#include "device.cuh"
#include "fused_schedule.cuh"
#include "kernels.h"
#include "wkv_tiles.cuh"

namespace engram {

namespace {

constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kXWarp = 2 + kEpiWarps;
constexpr int kGateWarp = kXWarp + 1;
constexpr int kFusedThreads = (kGateWarp + 1) * 32;
constexpr int kPairB = kBN / 2;            // wkv rows of a key tile staged by each CTA of a pair
constexpr int kStageABytes = kBM * kBK * 2;
constexpr int kStageBBytes = kPairB * kBK * 2;
constexpr int kXCols = 64;                 // columns per x box (128 B per row: one swizzle row)
constexpr int kXBoxBytes = kBM * kXCols * 2;
constexpr int kItemSlots = 4;              // item ring depth
// readers of an item slot: MMA issuer, x producer, gate warp and 8 epilogue warps in the even
// CTA; operand producer, x producer, gate warp and 8 epilogue warps in the odd CTA
constexpr int kItemReaders = 2 * (3 + kEpiWarps);
constexpr int kMaxHc = 8;
constexpr int kMaxFusedDim = 5120;
constexpr int kTokensPerTile = 2 * kBM;    // tokens per item
constexpr uint32_t kEpiBarrier = 1;        // named barrier of the epilogue warps

// Depths of the two shared-memory rings: operand stages (A and B of the pair MMA) and x slots.
// With the gate in the epilogue, value items stream x in and out through the x slots; with the
// output deferred only key items read x, and the same shared memory holds one more operand stage
// (measured 3% faster at 512-2048 tokens, where the operand loads wait on HBM).
struct RingsFused {
  static constexpr int kStages = 5;
  static constexpr int kXSlots = 4;
};
struct RingsDeferred {
  static constexpr int kStages = 6;
  static constexpr int kXSlots = 2;
};

template <class R>
struct FusedShared {
  uint64_t full[R::kStages];      // even CTA: operands of both CTAs landed
  uint64_t empty[R::kStages];     // both CTAs: the pair MMAs are done with the stage
  uint64_t tfull[2];              // both CTAs: accumulator ready
  uint64_t tempty[2];             // even CTA: both CTAs' epilogues released the accumulator
  uint64_t xfull[R::kXSlots];
  uint64_t xempty[R::kXSlots];
  uint64_t ifull[kItemSlots];     // both CTAs: item index written (by the even CTA's producer)
  uint64_t iempty[kItemSlots];    // even CTA: every reader of both CTAs has read the slot
  uint64_t pfull[2];              // a key tile's partial sums are in global memory (128 arrivals)
  uint64_t pempty[2];             // the gate warp has taken them
  uint64_t drain;
  int32_t item[kItemSlots];       // item index, or -1: no more items
  uint32_t tmem_base;
  int abort;
  // second-half partial sums, handed to the first half; one buffer suffices because the epilogue
  // warps meet at a barrier after the first half has read it and before the next key tile
  float part[3][kBM];
};

template <class R>
constexpr size_t fused_smem_bytes() {
  return size_t(R::kStages) * (kStageABytes + kStageBBytes) + size_t(R::kXSlots) * kXBoxBytes +
         sizeof(FusedShared<R>) + 1024;
}
static_assert(fused_smem_bytes<RingsFused>() <= 232448, "fused kernel exceeds 227 KB");
static_assert(fused_smem_bytes<RingsDeferred>() <= 232448, "fused kernel exceeds 227 KB");

struct FusedParams {
  const uint16_t* q;
  const uint16_t* k;
  const uint8_t* mask;
  uint16_t* out;
  float* gate_out;
  uint16_t* kv_out;
  uint16_t* vout;     // [M, dim] value rows (deferred output), or null
  float* gx;          // [M, hc] gates, exchanged between pairs
  float* part;        // [m_tiles, 2, hc, nk, 3, 128] per-key-tile partial sums
  int32_t* next;      // item counter; zero at launch
  int32_t* count;     // [m_tiles, 2, hc] key tiles done; zero at launch
  int32_t* flags;     // [m_tiles, 2, hc] 1 once the gates are in gx; zero at launch
  int64_t M;
  int32_t K, hc, dim;
  float eps, inv_sqrt_dim;
  uint32_t* err;
  LenAdvance adv;
  FusedSchedule sched;
};

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

template <int kWords>
__device__ __forceinline__ void store_words(uint16_t* p, const uint32_t* v) {
  uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int i = 0; i < kWords / 4; ++i)
    q[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

// Half a row (32 bf16 = 64 B) of a 128B-swizzled x box: 16-byte chunk j of row r sits at chunk
// position j ^ (r % 8); this half holds chunks 4*half .. 4*half + 3.
__device__ __forceinline__ void read_x_half_row(const uint8_t* box, int row, int half,
                                                uint32_t (&v)[16]) {
  const uint32_t base = smem_u32(box) + row * 128;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint4 t = lds128(base + (((4 * half + j) ^ (row & 7)) << 4));
    v[4 * j + 0] = t.x;
    v[4 * j + 1] = t.y;
    v[4 * j + 2] = t.z;
    v[4 * j + 3] = t.w;
  }
}

__device__ __forceinline__ void write_x_half_row(uint8_t* box, int row, int half,
                                                 const uint32_t (&v)[16]) {
  const uint32_t base = smem_u32(box) + row * 128;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    sts128(base + (((4 * half + j) ^ (row & 7)) << 4),
           make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
}

// Consumer side of the x ring. release() hands a slot back to the x producer: the proxy fence
// orders this thread's reads of the slot before the TMA load that will overwrite it.
template <int kSlots>
struct XRing {
  uint32_t slot = 0, phase = 0;
  __device__ __forceinline__ void advance() {
    if (++slot == kSlots) {
      slot = 0;
      phase ^= 1u;
    }
  }
  __device__ __forceinline__ void release(uint64_t* xempty) {
    fence_proxy_async_shared();
    mbar_arrive(&xempty[slot]);
    advance();
  }
};

__device__ __forceinline__ void st_release_gpu(int32_t* p, int32_t v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int32_t ld_acquire_gpu(const int32_t* p) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Wait until flags[j] == 1 for the hc flags of one token half; bounded (kWaitLimitNs), then the
// error bit and *abort are set.
__device__ bool wait_flags(const int32_t* flags, int hc, volatile int* abort, uint32_t* err) {
  const uint64_t t0 = globaltimer_ns();
  for (int j = 0; j < hc; ++j) {
    while (ld_acquire_gpu(flags + j) != 1) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort = 1;
        set_error(err, kErrWaitTimeout);
        return false;
      }
      __nanosleep(64);
    }
  }
  return true;
}

// barrier.red.or over the epilogue warps (non-aligned: every thread counted on its own): a
// barrier that also tells every thread whether any of them passed `pred`.
__device__ __forceinline__ bool epi_any(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "barrier.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(kEpiBarrier), "r"(kEpiThreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void st_cluster_s32(uint32_t addr, int32_t v) {
  asm volatile("st.shared::cluster.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ int32_t atom_add_acq_rel_gpu(int32_t* p, int32_t v) {
  int32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}

// Reader side of the item ring. next() waits (bounded) for the slot and reads the item; release()
// tells the even CTA's producer that this reader is done with the slot.
struct ItemReader {
  uint32_t slot = 0, phase = 0;
  template <class Sh>
  __device__ __forceinline__ bool next(Sh* sh, int32_t& item, volatile int* abort,
                                       uint32_t* err) {
    if (!mbar_wait<true>(&sh->ifull[slot], phase, abort, err)) return false;
    item = *reinterpret_cast<volatile int32_t*>(&sh->item[slot]);
    return true;
  }
  __device__ __forceinline__ void advance() {
    if (++slot == kItemSlots) {
      slot = 0;
      phase ^= 1u;
    }
  }
  __device__ __forceinline__ void release(uint32_t iempty_leader0) {
    mbar_arrive_remote(iempty_leader0 + slot * static_cast<uint32_t>(sizeof(uint64_t)));
    advance();
  }
};

// Column tile of wkv (in units of 256 rows) that an item multiplies with.
__device__ __forceinline__ int32_t wkv_tile(const FusedItem& it, int32_t key_tiles) {
  return it.value ? key_tiles + it.col : it.col;
}

template <class R>
__global__ void __launch_bounds__(kFusedThreads, 1)
    engram_fused_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmW,
                        const __grid_constant__ CUtensorMap tmX,
                        const __grid_constant__ CUtensorMap tmOut, const FusedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint8_t* sA = smem;
  constexpr int kFusedStages = R::kStages;
  constexpr int kXSlots = R::kXSlots;
  uint8_t* sB = sA + kFusedStages * kStageABytes;
  uint8_t* sX = sB + kFusedStages * kStageBBytes;
  FusedShared<R>* sh = reinterpret_cast<FusedShared<R>*>(sX + kXSlots * kXBoxBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t half_m = static_cast<int32_t>(cluster_ctarank());   // which 128 tokens
  const bool leader = half_m == 0;                                   // issues the pair's MMAs
  const uint16_t pair_mask = 3u;
  const int32_t hc = p.hc, dim = p.dim;
  const int32_t nk = dim / kBN;             // key tiles per stream (and value tiles)
  const int32_t key_tiles = hc * nk;        // key tiles per token tile
  const int kblocks = p.K / kBK;
  const FusedSchedule& sched = p.sched;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kFusedStages; ++i) {
      mbar_init(&sh->full[i], 1);
      mbar_init(&sh->empty[i], 1);
    }
    for (int i = 0; i < kXSlots; ++i) {
      mbar_init(&sh->xfull[i], 1);
      mbar_init(&sh->xempty[i], kEpiThreads);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->tfull[a], 1);
      mbar_init(&sh->tempty[a], 2 * kEpiThreads);
    }
    for (int i = 0; i < kItemSlots; ++i) {
      mbar_init(&sh->ifull[i], 1);
      mbar_init(&sh->iempty[i], kItemReaders);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh->pfull[i], kBM);
      mbar_init(&sh->pempty[i], 1);
    }
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmOut);
  }
  if (warp == 1) {
    tmem_alloc_pair(&sh->tmem_base, kTmemCols);   // collectively with the other CTA of the pair
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();   // both CTAs' barriers initialised before any cross-CTA arrival
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;
  volatile int* abort = &sh->abort;
  const uint32_t iempty_leader0 = map_to_rank(smem_u32(&sh->iempty[0]), 0);
  pdl_wait();   // rows (and the cache lengths) come from the previous kernel of the stream
  if (p.adv.len != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < 32)
    for (int32_t b = threadIdx.x; b < p.adv.B; b += 32)
      p.adv.len[b] = min(p.adv.len[b] + p.adv.T, p.adv.cap);

  if (warp == 0) {
    // ------------------------------------------------------------- GEMM operand producer
    if (lane == 0) {
      TmaRingT<kFusedStages> ring;
      const uint32_t leader_bar0 = map_to_rank(smem_u32(&sh->full[0]), 0);
      const uint32_t peer_item0 = map_to_rank(smem_u32(&sh->item[0]), 1);
      const uint32_t peer_ifull0 = map_to_rank(smem_u32(&sh->ifull[0]), 1);
      // every rows tile is read by (hc + 1) * dim / 256 items and every wkv tile by one item per
      // token tile: keep them in L2 ahead of the streamed x and out
      const uint64_t keep_l2 = l2_evict_last_policy();
      ItemReader ir;   // the odd CTA reads its items; the even CTA writes both rings
      uint32_t islot = 0, iphase = 0;
      for (;;) {
        int32_t idx;
        if (leader) {
          // the next item, taken only now (the operand ring still holds several K-blocks of the
          // current one, which hides the atomic's latency), so that a pair holds few items
          if (!mbar_wait<true>(&sh->iempty[islot], iphase ^ 1u, abort, p.err)) break;
          const int32_t got = atomicAdd(p.next, 1);
          idx = got < sched.items ? got : -1;
          sh->item[islot] = idx;
          st_cluster_s32(peer_item0 + islot * 4u, idx);
          mbar_arrive(&sh->ifull[islot]);
          mbar_arrive_remote(peer_ifull0 + islot * static_cast<uint32_t>(sizeof(uint64_t)));
          if (++islot == kItemSlots) {
            islot = 0;
            iphase ^= 1u;
          }
          if (idx < 0) break;
        } else {
          if (!ir.next(sh, idx, abort, p.err)) break;
          ir.release(iempty_leader0);
          if (idx < 0) break;
        }
        const FusedItem it = fused_item_at(sched, idx);
        const int32_t m0 = it.mt * kTokensPerTile + half_m * kBM;
        const int32_t n0 = wkv_tile(it, key_tiles) * kBN + half_m * kPairB;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ring.acquire(sh->empty, abort, p.err)) { ok = false; break; }
          const uint32_t full_bar =
              leader_bar0 + ring.stage * static_cast<uint32_t>(sizeof(uint64_t));
          if (leader)
            mbar_arrive_expect_tx(&sh->full[ring.stage], 2 * (kStageABytes + kStageBBytes));
          tma_load_2d_pair_hint(sA + ring.stage * kStageABytes, &tmA, full_bar, kb * kBK, m0,
                                keep_l2);
          tma_load_2d_pair_hint(sB + ring.stage * kStageBBytes, &tmW, full_bar, kb * kBK, n0,
                                keep_l2);
          ring.issued();
        }
        if (!ok) break;
      }
      // the even CTA's full barriers count this CTA's loads; it waits on them for both
      if (leader) ring.drain(sh->full);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer (even CTA)
    if (lane == 0 && leader) {
      uint32_t stage = 0, phase = 0, t_all = 0;
      ItemReader ir;
      const uint32_t idesc = idesc_bf16_f32(2 * kBM, kBN);
      for (;; ++t_all) {
        int32_t idx;
        if (!ir.next(sh, idx, abort, p.err)) break;
        ir.release(iempty_leader0);
        if (idx < 0) break;
        const uint32_t acc = t_all & 1, acc_phase = (t_all >> 1) & 1;
        if (!mbar_wait<true>(&sh->tempty[acc], acc_phase ^ 1u, abort, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * kBN;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&sh->full[stage], phase, abort, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad = sw128_kmajor_desc(smem_u32(sA + stage * kStageABytes));
          const uint64_t bd = sw128_kmajor_desc(smem_u32(sB + stage * kStageBBytes));
#pragma unroll
          for (int kk = 0; kk < kBK / kUmmaK; ++kk)
            tc_mma_bf16_pair(d, ad + 2ull * kk, bd + 2ull * kk, idesc, (kb | kk) != 0);
          tc_commit_pair_mc(&sh->empty[stage], pair_mask);
          if (++stage == kFusedStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit_pair_mc(&sh->tfull[acc], pair_mask);
      }
      tc_commit_pair_mc(&sh->drain, pair_mask);
    }
    // every pair MMA writing this CTA's TMEM has finished before TMEM is released
    if (lane == 0) mbar_wait_drain(&sh->drain, 0);
    __syncwarp();
  } else if (warp == kXWarp) {
    // ------------------------------------------------------------- x producer
    // Same order as the epilogue: a key item takes its stream's 4 boxes; a value item, for each
    // 64-column box of the tile, the hc streams in turn.
    if (lane == 0) {
      TmaRingT<kXSlots> ring;
      ItemReader ir;
      const uint64_t stream_l2 = l2_evict_first_policy();   // x: read by one key and one value item
      bool ok = true;
      while (ok) {
        int32_t idx;
        if (!ir.next(sh, idx, abort, p.err)) break;
        ir.release(iempty_leader0);
        if (idx < 0) break;
        const FusedItem it = fused_item_at(sched, idx);
        const int32_t m0 = it.mt * kTokensPerTile + half_m * kBM;
        // (deferred output: a value item reads no x)
        const int steps = it.value ? (p.vout ? 0 : (kBN / kXCols) * hc) : kBN / kXCols;
        for (int q = 0; q < steps; ++q) {
          int32_t col, stream;
          if (it.value) {
            col = it.col * kBN + (q / hc) * kXCols;
            stream = q % hc;
          } else {
            col = (it.col % nk) * kBN + q * kXCols;
            stream = it.col / nk;
          }
          if (!ring.acquire(sh->xempty, abort, p.err)) { ok = false; break; }
          mbar_arrive_expect_tx(&sh->xfull[ring.stage], kXBoxBytes);
          tma_load_3d_hint(sX + ring.stage * kXBoxBytes, &tmX, &sh->xfull[ring.stage], col,
                           stream, m0, stream_l2);
          ring.issued();
        }
      }
      ring.drain(sh->xfull);
    }
  } else if (warp == kGateWarp) {
    // ------------------------------------------------------------- gate warp
    // For every key tile this CTA finishes: count it in; if it was the last of its (token tile,
    // half, stream), add the partial sums of all the stream's key tiles in column order, form
    // the 128 gates and publish them.
    ItemReader ir;
    uint32_t nkey = 0;
    for (;;) {
      int32_t idx = -1;
      bool ok = ir.next(sh, idx, abort, p.err);
      ok = __all_sync(0xFFFFFFFFu, ok);
      __syncwarp();
      if (lane == 0) ir.release(iempty_leader0);
      else ir.advance();
      if (!ok || idx < 0) break;
      const FusedItem it = fused_item_at(sched, idx);
      if (it.value) continue;
      const uint32_t b = nkey & 1, ph = (nkey >> 1) & 1;
      ++nkey;
      ok = mbar_wait(&sh->pfull[b], ph, abort, p.err);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (!ok) break;
      const int32_t s = it.col / nk;
      const int64_t ts = (static_cast<int64_t>(it.mt) * 2 + half_m) * hc + s;
      int32_t last = 0;
      if (lane == 0) {
        __threadfence();   // the epilogue's partial sums (ordered before pfull) before the count
        last = atom_add_acq_rel_gpu(p.count + ts, 1) == nk - 1;
        mbar_arrive(&sh->pempty[b]);
      }
      last = __shfl_sync(0xFFFFFFFFu, last, 0);
      if (!last) continue;
      __threadfence();
      const float* pp = p.part + ts * nk * 3 * kBM;
      for (int r4 = 0; r4 < kBM / 32; ++r4) {
        const int rr = r4 * 32 + lane;
        const int64_t m = static_cast<int64_t>(it.mt) * kTokensPerTile + half_m * kBM + rr;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f;
        for (int j = 0; j < nk; ++j) {   // column order: independent of who ran what
          const float* pj = pp + static_cast<int64_t>(j) * 3 * kBM;
          a0 += __ldcg(pj + rr);
          a1 += __ldcg(pj + kBM + rr);
          a2 += __ldcg(pj + 2 * kBM + rr);
        }
        if (m < p.M) {
          const bool keep = p.mask == nullptr || p.mask[m] != 0;
          const float g = keep ? gate_from_sums(a0, a1, a2, dim, p.eps, p.inv_sqrt_dim) : 0.f;
          p.gx[m * hc + s] = g;
          if (p.gate_out) p.gate_out[m * hc + s] = g;
        }
      }
      __syncwarp();
      if (lane == 0) {
        __threadfence();
        st_release_gpu(p.flags + (static_cast<int64_t>(it.mt) * 2 + half_m) * hc + s, 1);
      }
    }
  } else {
    // ------------------------------------------------------------- epilogue (warps 2-9)
    // Failed waits (abort) are made warp-uniform at once and epilogue-uniform at the barriers, so
    // that every epilogue thread passes the same named barriers and leaves the loop together.
    const int quad = warp & 3;                       // TMEM lane quadrant
    const int half = (warp - 2) >> 2;                // which 32 columns of each 64-column box
    const int row = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const int64_t N = static_cast<int64_t>(dim) * (hc + 1);
    const uint32_t tempty_leader0 = map_to_rank(smem_u32(&sh->tempty[0]), 0);
    XRing<kXSlots> xr;
    // out is written once and read by nothing of this kernel: its lines go first (measured 0.5%
    // faster at 4096 and 16384 tokens than the default policy)
    const uint64_t out_l2 = l2_evict_first_policy();
    ItemReader ir;
    uint32_t nkey = 0;
    int32_t pending = -1;   // thread 64: x slot whose TMA store may still be reading it

    for (uint32_t t_all = 0;; ++t_all) {
      int32_t idx = -1;
      bool ok = ir.next(sh, idx, abort, p.err);
      ok = __all_sync(0xFFFFFFFFu, ok);
      __syncwarp();   // one arrival per warp, after every lane has read the item
      if (lane == 0) ir.release(iempty_leader0);
      else ir.advance();
      if (epi_any(!ok || idx < 0)) break;

      const FusedItem it = fused_item_at(sched, idx);
      const int64_t m = static_cast<int64_t>(it.mt) * kTokensPerTile + half_m * kBM + row;
      const bool valid = m < p.M;
      const bool keep = valid && (p.mask == nullptr || p.mask[m] != 0);
      int32_t* fl = p.flags + (static_cast<int64_t>(it.mt) * 2 + half_m) * hc;
      float gl[kMaxHc];
#pragma unroll
      for (int i = 0; i < kMaxHc; ++i) gl[i] = 0.f;
      if (it.value && p.vout == nullptr) {
        // the gates of every stream of these tokens (bounded wait)
        bool got = true;
        if (threadIdx.x == 64) got = wait_flags(fl, hc, abort, p.err);
        if (epi_any(!got)) break;
        if (valid) {
          ld_acquire_gpu(fl);   // this thread's own acquire of the published gates
#pragma unroll
          for (int i = 0; i < kMaxHc; ++i) gl[i] = i < hc ? __ldcg(p.gx + m * hc + i) : 0.f;
        }
      }

      const int32_t s = it.col / nk;                 // key item: its stream
      // w = q * k of the key tile's 256 columns (a product of two bf16 values, exact in f32):
      // lane l forms those of columns 8 l .. 8 l + 7 from one 16-byte load of q and one of k,
      // issued before the accumulator wait; each box then takes its 32 columns from the lanes
      // that hold them by broadcast shuffles
      float w8[8];
      if (!it.value) {
        const int64_t q0 = static_cast<int64_t>(s) * dim + (it.col % nk) * kBN + 8 * lane;
        const uint4 qa = __ldg(reinterpret_cast<const uint4*>(p.q + q0));
        const uint4 ka = __ldg(reinterpret_cast<const uint4*>(p.k + q0));
        const uint32_t qw[4] = {qa.x, qa.y, qa.z, qa.w}, kw[4] = {ka.x, ka.y, ka.z, ka.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          w8[2 * e] = lo_bf16(qw[e]) * lo_bf16(kw[e]);
          w8[2 * e + 1] = hi_bf16(qw[e]) * hi_bf16(kw[e]);
        }
      }

      const uint32_t acc = t_all & 1, acc_phase = (t_all >> 1) & 1;
      ok = mbar_wait(&sh->tfull[acc], acc_phase, abort, p.err);
      ok = __all_sync(0xFFFFFFFFu, ok);
      if (ok) tc_fence_after();
      const uint32_t tbase = tmem_base + lane_base + acc * kBN + half * 32;
      float sh2[2] = {0.f, 0.f}, sk2[2] = {0.f, 0.f}, shwk[2] = {0.f, 0.f};
      if (!it.value) {
        // key tile: columns d0 .. d0 + 255 of stream s, in four 64-column boxes
        for (int c4 = 0; c4 < kBN / kXCols && ok; ++c4) {
          const int32_t d = (it.col % nk) * kBN + c4 * kXCols + half * 32;   // this half's columns
          const int src0 = (c4 * kXCols + half * 32) / 8;   // lane holding the box-half's column 0
          uint32_t r[32];
          tc_ld_32x32b_x32(tbase + c4 * kXCols, r);
          ok = mbar_wait(&sh->xfull[xr.slot], xr.phase, abort, p.err);
          ok = __all_sync(0xFFFFFFFFu, ok);
          uint32_t xv[16];
          if (ok) read_x_half_row(sX + xr.slot * kXBoxBytes, row, half, xv);
          xr.release(sh->xempty);
          tc_wait_ld(r);
          if (!ok) break;
          uint32_t kb16[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            kb16[e] = pack_bf16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
            const float w0 = __shfl_sync(0xFFFFFFFFu, w8[(2 * e) % 8], src0 + (2 * e) / 8);
            const float w1 = __shfl_sync(0xFFFFFFFFu, w8[(2 * e + 1) % 8], src0 + (2 * e + 1) / 8);
            const float key0 = lo_bf16(kb16[e]), key1 = hi_bf16(kb16[e]);
            const float h0 = lo_bf16(xv[e]), h1 = hi_bf16(xv[e]);
            sh2[0] = fmaf(h0, h0, sh2[0]);
            sk2[0] = fmaf(key0, key0, sk2[0]);
            shwk[0] = fmaf(h0 * w0, key0, shwk[0]);
            sh2[1] = fmaf(h1, h1, sh2[1]);
            sk2[1] = fmaf(key1, key1, sk2[1]);
            shwk[1] = fmaf(h1 * w1, key1, shwk[1]);
          }
          if (valid && p.kv_out)
            store_words<16>(p.kv_out + m * N + static_cast<int64_t>(s) * dim + d, kb16);
        }
      } else if (p.vout != nullptr) {
        // value tile, deferred output: the bf16 value rows only; a later kernel adds
        // gate * value to x once every gate exists, so this item waits for no key tile
        const int32_t col0 = it.col * kBN;
        for (int c4 = 0; c4 < kBN / kXCols && ok; ++c4) {
          const int32_t colb = col0 + c4 * kXCols + half * 32;
          uint32_t r[32];
          tc_ld_32x32b_x32(tbase + c4 * kXCols, r);
          tc_wait_ld(r);
          uint32_t vb[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            vb[e] = pack_bf16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
          if (valid) {
            store_words<16>(p.vout + m * dim + colb, vb);
            if (p.kv_out)
              store_words<16>(p.kv_out + m * N + static_cast<int64_t>(hc) * dim + colb, vb);
          }
        }
      } else {
        // value tile: value columns col0 .. col0 + 255, shared by all hc streams. Each (64-column
        // box, stream) is computed in place in its x slot and written out by one TMA store; the
        // slot goes back to the x producer once the store has read it.
        const int32_t col0 = it.col * kBN;
        const int32_t m0 = it.mt * kTokensPerTile + half_m * kBM;
        for (int c4 = 0; c4 < kBN / kXCols && ok; ++c4) {
          const int32_t colb = col0 + c4 * kXCols;
          uint32_t r[32];
          tc_ld_32x32b_x32(tbase + c4 * kXCols, r);
          tc_wait_ld(r);
          uint32_t vb[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            vb[e] = pack_bf16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
          if (valid && p.kv_out)
            store_words<16>(p.kv_out + m * N + static_cast<int64_t>(hc) * dim + colb + half * 32,
                            vb);
          for (int s2 = 0; s2 < hc; ++s2) {
            ok = mbar_wait(&sh->xfull[xr.slot], xr.phase, abort, p.err);
            ok = __all_sync(0xFFFFFFFFu, ok);
            uint8_t* box = sX + xr.slot * kXBoxBytes;
            if (ok && keep) {   // a masked token's x passes through unchanged
              float g = gl[0];
#pragma unroll
              for (int i = 1; i < kMaxHc; ++i) g = (s2 == i) ? gl[i] : g;
              uint32_t xv[16];
              read_x_half_row(box, row, half, xv);
#pragma unroll
              for (int e = 0; e < 16; ++e)
                xv[e] = pack_bf16x2(fmaf(g, lo_bf16(vb[e]), lo_bf16(xv[e])),
                                    fmaf(g, hi_bf16(vb[e]), hi_bf16(xv[e])));
              write_x_half_row(box, row, half, xv);
            }
            fence_proxy_async_shared();   // the box's writes, before the TMA store reads them
            const bool fail = epi_any(!ok);
            if (threadIdx.x == 64) {
              if (!fail) {
                tma_store_3d_hint(&tmOut, box, colb, s2, m0, out_l2);
                bulk_commit_group();
              }
              bulk_wait_group_read<1>();   // every store but this one has read its slot
              if (pending >= 0) mbar_arrive(&sh->xempty[pending]);
              pending = static_cast<int32_t>(xr.slot);
            } else {
              mbar_arrive(&sh->xempty[xr.slot]);
            }
            xr.advance();
            if (fail) {
              ok = false;
              break;
            }
          }
        }
        if (threadIdx.x == 64 && pending >= 0) {
          bulk_wait_group_read<0>();
          mbar_arrive(&sh->xempty[pending]);
          pending = -1;
        }
      }
      // hand the accumulator back to the pair's MMA issuer
      tc_fence_before();
      mbar_arrive_remote(tempty_leader0 + acc * static_cast<uint32_t>(sizeof(uint64_t)));

      if (!it.value) {
        // The key tile's sums: the second half hands its partial sums to the first, which writes
        // this CTA's 128 rows of them to the partial buffer and hands the tile to the gate warp.
        const uint32_t b = nkey & 1, ph = (nkey >> 1) & 1;
        ++nkey;
        if (half == 1) {
          sh->part[0][row] = sh2[0] + sh2[1];
          sh->part[1][row] = sk2[0] + sk2[1];
          sh->part[2][row] = shwk[0] + shwk[1];
        }
        if (epi_any(!ok)) break;
        if (half == 0) {
          const int64_t ts = (static_cast<int64_t>(it.mt) * 2 + half_m) * hc + s;
          float* pj = p.part + (ts * nk + it.col % nk) * 3 * kBM;
          __stcg(pj + row, sh2[0] + sh2[1] + sh->part[0][row]);
          __stcg(pj + kBM + row, sk2[0] + sk2[1] + sh->part[1][row]);
          __stcg(pj + 2 * kBM + row, shwk[0] + shwk[1] + sh->part[2][row]);
          ok = mbar_wait(&sh->pempty[b], ph ^ 1u, abort, p.err);
          ok = __all_sync(0xFFFFFFFFu, ok);
          if (ok) mbar_arrive(&sh->pfull[b]);
        }
      }
      if (epi_any(!ok)) break;
    }
    if (threadIdx.x == 64) bulk_wait_group<0>();   // the output stores are complete
  }

  // The pair's TMEM is released by both CTAs together, so neither may do so while the other
  // still reads its accumulators: both CTAs finish (all their waits are bounded) first.
  tc_fence_before();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);   // collectively with the other CTA of the pair
  }
}

// Largest number of CTA pairs of this kernel that can be resident at once on the current device
// (the kernel's shared-memory limit must have been raised first).
int query_resident_pairs() {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kFusedThreads, 1, 1);
  cfg.dynamicSmemBytes = fused_smem_bytes<RingsFused>();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, engram_fused_kernel<RingsFused>, &cfg) != cudaSuccess ||
      n <= 0)
    n = 1;
  return n;
}

int max_resident_pairs() { return fused_resident_pairs_cached(query_resident_pairs); }

size_t round256(size_t n) { return (n + 255) & ~size_t(255); }

struct ScratchLayout {
  size_t gx, part, sync, sync_bytes, total;
};

// gx [M, hc] f32 | partial sums [m_tiles, 2, hc, nk, 3, 128] f32 |
// item counter, then count and flags [m_tiles, 2, hc] each (int32, cleared before each launch)
ScratchLayout scratch_layout(int64_t M, int32_t hc, int32_t dim) {
  const int64_t m_tiles = (M + kTokensPerTile - 1) / kTokensPerTile;
  ScratchLayout l{};
  l.gx = 0;
  l.part = round256(size_t(M) * hc * 4);
  l.sync = l.part + round256(size_t(m_tiles) * 2 * hc * (dim / kBN) * 3 * kBM * 4);
  l.sync_bytes = (1 + size_t(m_tiles) * 2 * hc * 2) * 4;
  l.total = l.sync + round256(l.sync_bytes);
  return l;
}

}  // namespace

bool fused_supported(int32_t K, int32_t hc, int32_t dim) {
  return K > 0 && K % kBK == 0 && hc >= 1 && hc <= kMaxHc && dim % kBN == 0 &&
         dim <= kMaxFusedDim;
}

size_t fused_scratch_bytes(int64_t M, int32_t hc, int32_t dim) {
  return scratch_layout(M, hc, dim).total;
}

const float* fused_gates(const void* scratch) {
  return reinterpret_cast<const float*>(static_cast<const uint8_t*>(scratch));   // layout: gx first
}

void fused_sync_region(void* scratch, int64_t M, int32_t hc, int32_t dim, int32_t** ptr,
                       int32_t* count) {
  const ScratchLayout l = scratch_layout(M, hc, dim);
  *ptr = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(scratch) + l.sync);
  *count = static_cast<int32_t>(l.sync_bytes / 4);
}

cudaError_t launch_fused(const FusedArgs& a, cudaStream_t st, bool pdl) {
  const int64_t N = static_cast<int64_t>(a.dim) * (a.hc + 1);
  const int64_t m_tiles = (a.M + kTokensPerTile - 1) / kTokensPerTile;
  alignas(64) CUtensorMap tmA, tmW, tmX, tmOut;
  if (!tensor_map_2d_bf16(&tmA, a.a, a.K, a.M, kBK, kBM) ||
      !tensor_map_2d_bf16(&tmW, a.w, a.K, N, kBK, kPairB) ||
      !tensor_map_3d_bf16(&tmX, a.x, a.dim, a.hc, a.M, kXCols, 1, kBM) ||
      !tensor_map_3d_bf16(&tmOut, a.out, a.dim, a.hc, a.M, kXCols, 1, kBM))
    return cudaErrorInvalidValue;
  // the deferred output (value rows stored, no x for value items) takes the deeper operand ring
  const bool deferred = a.vout != nullptr;
  const void* kernel = deferred
                           ? reinterpret_cast<const void*>(engram_fused_kernel<RingsDeferred>)
                           : reinterpret_cast<const void*>(engram_fused_kernel<RingsFused>);
  const size_t smem = deferred ? fused_smem_bytes<RingsDeferred>() : fused_smem_bytes<RingsFused>();
  {
    // the resident-pairs query below runs on the fused-output kernel: raise its limit in any case
    cudaError_t e = ensure_dynamic_smem(
        reinterpret_cast<const void*>(engram_fused_kernel<RingsFused>),
        fused_smem_bytes<RingsFused>());
    if (e == cudaSuccess && deferred) e = ensure_dynamic_smem(kernel, smem);
    if (e != cudaSuccess) return e;
  }
  const ScratchLayout l = scratch_layout(a.M, a.hc, a.dim);
  uint8_t* base = static_cast<uint8_t*>(a.scratch);
  int32_t* sync = reinterpret_cast<int32_t*>(base + l.sync);
  if (!a.sync_cleared) {
    cudaError_t e = cudaMemsetAsync(sync, 0, l.sync_bytes, st);
    if (e != cudaSuccess) return e;
  }

  const int32_t nk = a.dim / kBN;
  const int64_t items = m_tiles * (int64_t(a.hc) * nk + nk);
  int64_t pairs = max_resident_pairs();
  if (pairs > items) pairs = items;

  FusedParams p{};
  p.q = a.q;
  p.k = a.k;
  p.mask = a.mask;
  p.out = a.out;
  p.gate_out = a.gate_out;
  p.kv_out = a.kv_out;
  p.vout = a.vout;
  p.gx = reinterpret_cast<float*>(base + l.gx);
  p.part = reinterpret_cast<float*>(base + l.part);
  p.next = sync;
  p.count = sync + 1;
  p.flags = sync + 1 + m_tiles * 2 * a.hc;
  p.M = a.M;
  p.K = a.K;
  p.hc = a.hc;
  p.dim = a.dim;
  p.eps = a.eps;
  p.inv_sqrt_dim = a.inv_sqrt_dim;
  p.err = a.err;
  p.adv = a.adv;
  p.sched = make_fused_schedule(m_tiles, a.hc * nk, nk, static_cast<int32_t>(pairs));

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2, static_cast<unsigned>(pairs), 1);
  cfg.blockDim = dim3(kFusedThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  // No co-residency is needed: a pair takes items only while it runs, and takes them in the
  // schedule's order, so every item a value item waits for is held by a running pair.
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // with the counters already cleared by the previous kernel, the launch and prologue overlap
  // it; the kernel waits for it before touching its data
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (pdl && a.sync_cleared) ? 2 : 1;
  if (deferred)
    return cudaLaunchKernelEx(&cfg, engram_fused_kernel<RingsDeferred>, tmA, tmW, tmX, tmOut, p);
  return cudaLaunchKernelEx(&cfg, engram_fused_kernel<RingsFused>, tmA, tmW, tmX, tmOut, p);
}

}  // namespace engram
