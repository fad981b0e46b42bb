// Stages 3 + 4 fused: the wkv projection on the tensor cores with the gate-and-add in its
// epilogue, so the dim * (hc + 1)-wide kv row never goes to HBM.
//
// Engram listing, forward: kv = wkv(rows); key, value = split(kv); per (token, stream) the three
// sums over dim (h^2, key^2, h*w*key) give the gate; out = bf16(h + gate * value).
//
// Work split. Tokens come in tiles of 256. For each tile and each stream s there is one CTA pair
// (a 2-CTA cluster): CTA h of the pair owns tokens [128h, 128h + 128) of the tile. Together the
// pair runs the projection as CTA-pair MMAs (tcgen05 cta_group::2, M = 256): each CTA stages its
// 128 rows of the gathered activations and half of the 256 wkv rows of a tile per K-block, and
// receives its 128 x 256 accumulator in its own TMEM. This halves the shared-memory operand
// traffic per SM of a single-CTA 128 x 256 MMA. The even CTA issues the MMAs; both CTAs' TMA
// loads count on its barriers and its commits arrive on the barriers of both.
//
// Pair s computes stream s's dim / 256 key tiles and accumulates sum h^2, sum key^2 and
// sum h*w*key for its tokens on its own (no partial sums cross CTAs). Each CTA then publishes its
// 128 gates to global memory with a release flag, and waits (bounded) for the gates of the other
// streams' pairs of the same tokens. Pair s then computes its share [s*dim/hc, (s+1)*dim/hc) of
// the value columns and writes out[m, s', cols] = h + gate[m, s'] * value for every stream s'.
// The pairs that exchange gates must run at the same time: the kernel is a cooperative launch
// (co-residency guaranteed) with a persistent loop over token tiles.
//
// Roles per CTA (352 threads):
//   warp 0       TMA producer of this CTA's half of the GEMM operands, 4-stage ring;
//   warp 1       TMEM owner; in the even CTA also the MMA issuer (two 256-column accumulators);
//   warps 2-9    epilogue: two warps per TMEM lane quadrant (warp w reads lanes 32*(w%4)...),
//                thread = (token row, half of each 64-column box): tcgen05.ld, gate sums, output;
//   warp 10      TMA producer of the residual streams x: 128-token x 64-column boxes into a
//                3-slot ring, in exactly the order the epilogue consumes them.
// w = q_weight[s] * k_weight[s] (f32, exact) is staged in shared memory once per CTA.
#include "device.cuh"
#include "kernels.h"
#include "wkv_tiles.cuh"

namespace engram {

namespace {

constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kXWarp = 2 + kEpiWarps;
constexpr int kFusedThreads = (kXWarp + 1) * 32;
constexpr int kFusedStages = 4;            // A/B ring depth
constexpr int kPairB = kBN / 2;            // wkv rows of a key tile staged by each CTA of a pair
constexpr int kStageABytes = kBM * kBK * 2;
constexpr int kStageBBytes = kPairB * kBK * 2;
constexpr int kXSlots = 3;                 // x ring depth
constexpr int kXCols = 64;                 // columns per x box (128 B per row: one swizzle row)
constexpr int kXBoxBytes = kBM * kXCols * 2;
constexpr int kMaxHc = 8;
constexpr int kMaxFusedDim = 5120;         // w tile in shared memory: dim floats
constexpr int kTokensPerTile = 2 * kBM;    // tokens per pair
constexpr uint32_t kEpiBarrier = 1;        // named barrier of the epilogue warps

struct FusedShared {
  uint64_t full[kFusedStages];    // even CTA: operands of both CTAs landed
  uint64_t empty[kFusedStages];   // both CTAs: the pair MMAs are done with the stage
  uint64_t tfull[2];              // both CTAs: accumulator ready
  uint64_t tempty[2];             // even CTA: both CTAs' epilogues released the accumulator
  uint64_t xfull[kXSlots];
  uint64_t xempty[kXSlots];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  float part[3][kBM];             // second-half partial sums, handed to the first half
};

size_t fused_smem_bytes(int dim) {
  return size_t(kFusedStages) * (kStageABytes + kStageBBytes) + size_t(kXSlots) * kXBoxBytes +
         size_t(dim) * sizeof(float) + sizeof(FusedShared) + 1024;
}

struct FusedParams {
  const uint16_t* q;
  const uint16_t* k;
  const uint8_t* mask;
  uint16_t* out;
  float* gate_out;
  uint16_t* kv_out;
  float* gx;          // [M, hc] gates, exchanged between the streams' pairs
  int32_t* flags;     // [tiles, 2, hc] set to 1 once a CTA's gates are in gx; zero at launch
  int64_t M;
  int32_t K, hc, dim, bnv, m_tiles;
  float eps, inv_sqrt_dim;
  uint32_t* err;
  LenAdvance adv;
};

// Value columns per stream are split into tiles of bnv columns: the largest multiple of 64 that
// divides dim / hc and is at most 256 (each CTA of a pair stages bnv / 2 wkv rows).
int value_tile_width(int32_t hc, int32_t dim) {
  if (hc <= 0 || dim % hc != 0) return 0;
  const int v = dim / hc;
  for (int w = 256; w >= 64; w -= 64)
    if (v % w == 0) return w;
  return 0;
}

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

// Consumer side of the x ring. release() hands a slot back to the x producer: the proxy fence
// orders this thread's reads of the slot before the TMA load that will overwrite it.
struct XRing {
  uint32_t slot = 0, phase = 0;
  __device__ __forceinline__ void release(uint64_t* xempty) {
    fence_proxy_async_shared();
    mbar_arrive(&xempty[slot]);
    if (++slot == kXSlots) {
      slot = 0;
      phase ^= 1u;
    }
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

__global__ void __launch_bounds__(kFusedThreads, 1)
    engram_fused_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmWk,
                        const __grid_constant__ CUtensorMap tmWv,
                        const __grid_constant__ CUtensorMap tmX, const FusedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = sA + kFusedStages * kStageABytes;
  uint8_t* sX = sB + kFusedStages * kStageBBytes;
  float* sW = reinterpret_cast<float*>(sX + kXSlots * kXBoxBytes);
  FusedShared* sh = reinterpret_cast<FusedShared*>(sW + p.dim);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t half_m = static_cast<int32_t>(cluster_ctarank());   // which 128 tokens
  const bool leader = half_m == 0;                                   // issues the pair's MMAs
  const uint16_t pair_mask = 3u;
  const int32_t s = static_cast<int32_t>(blockIdx.y);                // this pair's stream
  const int32_t hc = p.hc, dim = p.dim, bnv = p.bnv;
  const int32_t vcols = dim / hc;
  const int nk = dim / kBN;                 // key tiles
  const int nv = vcols / bnv;               // value tiles
  const int ntiles = nk + nv;
  const int kblocks = p.K / kBK;
  const int first_tile = static_cast<int>(blockIdx.z), tile_step = static_cast<int>(gridDim.z);

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
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmWk);
    tma_prefetch_desc(&tmWv);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    tmem_alloc_pair(&sh->tmem_base, kTmemCols);   // collectively with the other CTA of the pair
    tmem_relinquish_pair();
  }
  // w = q * k for this CTA's stream: a product of two bf16 values, exact in f32
  for (int d = threadIdx.x; d < dim; d += kFusedThreads) {
    const int64_t i = static_cast<int64_t>(s) * dim + d;
    sW[d] = bf16_bits_to_f32(__ldg(p.q + i)) * bf16_bits_to_f32(__ldg(p.k + i));
  }
  tc_fence_before();
  cluster_sync_all();   // both CTAs' barriers initialised before any cross-CTA arrival
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;
  volatile int* abort = &sh->abort;
  pdl_wait();   // rows (and the cache lengths) come from the previous kernel of the stream
  if (p.adv.len != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 &&
      threadIdx.x < 32)
    for (int32_t b = threadIdx.x; b < p.adv.B; b += 32)
      p.adv.len[b] = min(p.adv.len[b] + p.adv.T, p.adv.cap);

  if (warp == 0) {
    // ------------------------------------------------------------- GEMM operand producer
    if (lane == 0) {
      TmaRingT<kFusedStages> ring;
      const uint32_t leader_bar0 = map_to_rank(smem_u32(&sh->full[0]), 0);
      for (int mt = first_tile; mt < p.m_tiles && !*abort; mt += tile_step) {
        const int32_t m0 = mt * kTokensPerTile + half_m * kBM;
        for (int t = 0; t < ntiles && !*abort; ++t) {
          const bool key = t < nk;
          const int32_t nb = key ? kPairB : bnv / 2;          // wkv rows this CTA stages
          const int32_t n0 = (key ? s * dim + t * kBN : hc * dim + s * vcols + (t - nk) * bnv) +
                             half_m * nb;
          const uint32_t bytes = static_cast<uint32_t>(kStageABytes + nb * kBK * 2);
          for (int kb = 0; kb < kblocks; ++kb) {
            if (!ring.acquire(sh->empty, abort, p.err)) break;
            const uint32_t full_bar =
                leader_bar0 + ring.stage * static_cast<uint32_t>(sizeof(uint64_t));
            if (leader) mbar_arrive_expect_tx(&sh->full[ring.stage], 2 * bytes);
            tma_load_2d_pair(sA + ring.stage * kStageABytes, &tmA, full_bar, kb * kBK, m0);
            tma_load_2d_pair(sB + ring.stage * kStageBBytes, key ? &tmWk : &tmWv, full_bar,
                             kb * kBK, n0);
            ring.issued();
          }
        }
      }
      // the even CTA's full barriers count this CTA's loads; it waits on them for both
      if (leader) ring.drain(sh->full);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer (even CTA)
    if (lane == 0 && leader) {
      uint32_t stage = 0, phase = 0, t_all = 0;
      bool ok = true;
      for (int mt = first_tile; mt < p.m_tiles && ok && !*abort; mt += tile_step) {
        for (int t = 0; t < ntiles && ok && !*abort; ++t, ++t_all) {
          const uint32_t acc = t_all & 1, acc_phase = (t_all >> 1) & 1;
          if (!mbar_wait<true>(&sh->tempty[acc], acc_phase ^ 1u, abort, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + acc * kBN;
          const uint32_t idesc = idesc_bf16_f32(2 * kBM, t < nk ? kBN : bnv);
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
      }
      tc_commit_pair_mc(&sh->drain, pair_mask);
    }
    // every pair MMA writing this CTA's TMEM has finished before TMEM is released
    if (lane == 0) mbar_wait_drain(&sh->drain, 0);
    __syncwarp();
  } else if (warp == kXWarp) {
    // ------------------------------------------------------------- x producer
    // Same order as the epilogue, per token tile: key tiles (stream s, 4 boxes each), then value
    // tiles (for each 64-column box of the tile, the hc streams in turn).
    if (lane == 0) {
      TmaRingT<kXSlots> ring;
      const int steps = nk * (kBN / kXCols) + nv * (bnv / kXCols) * hc;
      for (int mt = first_tile; mt < p.m_tiles && !*abort; mt += tile_step) {
        const int32_t m0 = mt * kTokensPerTile + half_m * kBM;
        for (int q = 0; q < steps && !*abort; ++q) {
          int32_t col, stream;
          if (q < nk * (kBN / kXCols)) {
            col = q * kXCols;
            stream = s;
          } else {
            const int v = q - nk * (kBN / kXCols);
            col = s * vcols + (v / hc) * kXCols;
            stream = v % hc;
          }
          if (!ring.acquire(sh->xempty, abort, p.err)) break;
          mbar_arrive_expect_tx(&sh->xfull[ring.stage], kXBoxBytes);
          tma_load_3d(sX + ring.stage * kXBoxBytes, &tmX, &sh->xfull[ring.stage], col, stream,
                      m0);
          ring.issued();
        }
      }
      ring.drain(sh->xfull);
    }
  } else {
    // ------------------------------------------------------------- epilogue (warps 2-9)
    const int quad = warp & 3;                       // TMEM lane quadrant
    const int half = (warp - 2) >> 2;                // which 32 columns of each 64-column box
    const int row = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const int64_t N = static_cast<int64_t>(dim) * (hc + 1);
    const uint32_t tempty_leader0 = map_to_rank(smem_u32(&sh->tempty[0]), 0);
    XRing xr;
    uint32_t t_all = 0;
    bool ok = true;

    for (int mt = first_tile; mt < p.m_tiles && ok; mt += tile_step) {
      const int64_t m = static_cast<int64_t>(mt) * kTokensPerTile + half_m * kBM + row;
      const bool valid = m < p.M;
      const bool keep = valid && (p.mask == nullptr || p.mask[m] != 0);
      // two accumulators per sum shorten the dependent FMA chains
      float sh2[2] = {0.f, 0.f}, sk2[2] = {0.f, 0.f}, shwk[2] = {0.f, 0.f};
      float gl[kMaxHc];
#pragma unroll
      for (int i = 0; i < kMaxHc; ++i) gl[i] = 0.f;

      for (int t = 0; t < ntiles && ok; ++t, ++t_all) {
        const uint32_t acc = t_all & 1, acc_phase = (t_all >> 1) & 1;
        if (!mbar_wait(&sh->tfull[acc], acc_phase, abort, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tbase = tmem_base + lane_base + acc * kBN + half * 32;
        if (t < nk) {
          // key tile: columns d0 .. d0 + 255 of stream s, in four 64-column boxes
          for (int c4 = 0; c4 < kBN / kXCols; ++c4) {
            const int32_t d = t * kBN + c4 * kXCols + half * 32;   // first column of this half
            uint32_t r[32];
            tc_ld_32x32b_x32(tbase + c4 * kXCols, r);
            if (!mbar_wait(&sh->xfull[xr.slot], xr.phase, abort, p.err)) { ok = false; break; }
            uint32_t xv[16];
            read_x_half_row(sX + xr.slot * kXBoxBytes, row, half, xv);
            xr.release(sh->xempty);
            tc_wait_ld(r);
            uint32_t kb16[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              kb16[e] = pack_bf16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
              const float2 w2 = *reinterpret_cast<const float2*>(sW + d + 2 * e);
              const float key0 = lo_bf16(kb16[e]), key1 = hi_bf16(kb16[e]);
              const float h0 = lo_bf16(xv[e]), h1 = hi_bf16(xv[e]);
              sh2[0] = fmaf(h0, h0, sh2[0]);
              sk2[0] = fmaf(key0, key0, sk2[0]);
              shwk[0] = fmaf(h0 * w2.x, key0, shwk[0]);
              sh2[1] = fmaf(h1, h1, sh2[1]);
              sk2[1] = fmaf(key1, key1, sk2[1]);
              shwk[1] = fmaf(h1 * w2.y, key1, shwk[1]);
            }
            if (valid && p.kv_out)
              store_words<16>(p.kv_out + m * N + static_cast<int64_t>(s) * dim + d, kb16);
          }
        } else {
          // value tile: value columns col0 .. col0 + bnv - 1, shared by all hc streams
          const int32_t col0 = s * vcols + (t - nk) * bnv;
          for (int c4 = 0; c4 < bnv / kXCols && ok; ++c4) {
            const int32_t col = col0 + c4 * kXCols + half * 32;
            uint32_t r[32];
            tc_ld_32x32b_x32(tbase + c4 * kXCols, r);
            tc_wait_ld(r);
            uint32_t vb[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              vb[e] = pack_bf16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
            if (valid && p.kv_out)
              store_words<16>(p.kv_out + m * N + static_cast<int64_t>(hc) * dim + col, vb);
            for (int s2 = 0; s2 < hc; ++s2) {
              if (!mbar_wait(&sh->xfull[xr.slot], xr.phase, abort, p.err)) { ok = false; break; }
              uint32_t xv[16];
              read_x_half_row(sX + xr.slot * kXBoxBytes, row, half, xv);
              xr.release(sh->xempty);
              if (!valid) continue;
              if (keep) {
                float g = gl[0];
#pragma unroll
                for (int i = 1; i < kMaxHc; ++i) g = (s2 == i) ? gl[i] : g;
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  xv[e] = pack_bf16x2(fmaf(g, lo_bf16(vb[e]), lo_bf16(xv[e])),
                                      fmaf(g, hi_bf16(vb[e]), hi_bf16(xv[e])));
              }   // a masked token's x passes through unchanged
              store_words<16>(p.out + (m * hc + s2) * dim + col, xv);
            }
          }
        }
        if (!ok) break;
        // hand the accumulator back to the pair's MMA issuer
        tc_fence_before();
        mbar_arrive_remote(tempty_leader0 + acc * static_cast<uint32_t>(sizeof(uint64_t)));

        if (t == nk - 1) {
          // all key tiles done. The second half hands its partial sums to the first; the first
          // half forms the gates of this CTA's 128 tokens and publishes them; then everyone
          // waits for the gates of every stream for these tokens.
          const float a0 = sh2[0] + sh2[1], a1 = sk2[0] + sk2[1], a2 = shwk[0] + shwk[1];
          if (half == 1) {
            sh->part[0][row] = a0;
            sh->part[1][row] = a1;
            sh->part[2][row] = a2;
          }
          named_bar_sync(kEpiBarrier, kEpiThreads);
          if (half == 0) {
            float g = 0.f;
            if (keep)
              g = gate_from_sums(a0 + sh->part[0][row], a1 + sh->part[1][row],
                                 a2 + sh->part[2][row], dim, p.eps, p.inv_sqrt_dim);
            if (valid) {
              p.gx[m * hc + s] = g;
              if (p.gate_out) p.gate_out[m * hc + s] = g;
            }
          }
          int32_t* fl = p.flags + (static_cast<int64_t>(mt) * 2 + half_m) * hc;
          named_bar_sync(kEpiBarrier, kEpiThreads);   // every gate of this CTA is written
          if (threadIdx.x == 64) {
            __threadfence();
            st_release_gpu(fl + s, 1);
            wait_flags(fl, hc, abort, p.err);
          }
          named_bar_sync(kEpiBarrier, kEpiThreads);   // every stream's gates are visible
          if (*abort) { ok = false; break; }
          if (valid) {
            ld_acquire_gpu(fl);   // this thread's own acquire of the published gates
#pragma unroll
            for (int i = 0; i < kMaxHc; ++i) gl[i] = i < hc ? __ldcg(p.gx + m * hc + i) : 0.f;
          }
        }
      }
    }
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

int g_max_pairs = 0;

// Largest number of CTA pairs of this kernel that can be resident at once.
int max_resident_pairs() {
  if (g_max_pairs == 0) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kFusedThreads, 1, 1);
    cfg.dynamicSmemBytes = fused_smem_bytes(kMaxFusedDim);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, engram_fused_kernel, &cfg) != cudaSuccess || n <= 0)
      n = 1;
    g_max_pairs = n;
  }
  return g_max_pairs;
}

size_t round256(size_t n) { return (n + 255) & ~size_t(255); }

}  // namespace

bool fused_supported(int32_t K, int32_t hc, int32_t dim) {
  return K > 0 && K % kBK == 0 && hc >= 1 && hc <= kMaxHc && dim % kBN == 0 &&
         dim <= kMaxFusedDim && value_tile_width(hc, dim) > 0;
}

size_t fused_scratch_bytes(int64_t M, int32_t hc) {
  const int64_t tiles = (M + kTokensPerTile - 1) / kTokensPerTile;
  return round256(size_t(M) * hc * 4) + round256(size_t(tiles) * 2 * hc * 4);
}

cudaError_t launch_fused(const FusedArgs& a, cudaStream_t st, bool /*pdl*/) {
  const int bnv = value_tile_width(a.hc, a.dim);
  const int64_t N = static_cast<int64_t>(a.dim) * (a.hc + 1);
  const int64_t m_tiles = (a.M + kTokensPerTile - 1) / kTokensPerTile;
  alignas(64) CUtensorMap tmA, tmWk, tmWv, tmX;
  if (!tensor_map_2d_bf16(&tmA, a.a, a.K, a.M, kBK, kBM) ||
      !tensor_map_2d_bf16(&tmWk, a.w, a.K, N, kBK, kPairB) ||
      !tensor_map_2d_bf16(&tmWv, a.w, a.K, N, kBK, bnv / 2) ||
      !tensor_map_3d_bf16(&tmX, a.x, a.dim, a.hc, a.M, kXCols, 1, kBM))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(engram_fused_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(fused_smem_bytes(kMaxFusedDim)));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  // scratch: the exchanged gates, then the flags (cleared before the launch)
  float* gx = static_cast<float*>(a.scratch);
  int32_t* flags = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(a.scratch) +
                                              round256(size_t(a.M) * a.hc * 4));
  cudaError_t e = cudaMemsetAsync(flags, 0, size_t(m_tiles) * 2 * a.hc * 4, st);
  if (e != cudaSuccess) return e;

  FusedParams p{};
  p.q = a.q;
  p.k = a.k;
  p.mask = a.mask;
  p.out = a.out;
  p.gate_out = a.gate_out;
  p.kv_out = a.kv_out;
  p.gx = gx;
  p.flags = flags;
  p.M = a.M;
  p.K = a.K;
  p.hc = a.hc;
  p.dim = a.dim;
  p.bnv = bnv;
  p.m_tiles = static_cast<int32_t>(m_tiles);
  p.eps = a.eps;
  p.inv_sqrt_dim = a.inv_sqrt_dim;
  p.err = a.err;
  p.adv = a.adv;

  // persistent: slots of token tiles with hc pairs each, all resident together
  int64_t slots = max_resident_pairs() / a.hc;
  if (slots < 1) return cudaErrorNotSupported;
  if (slots > m_tiles) slots = m_tiles;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2, static_cast<unsigned>(a.hc), static_cast<unsigned>(slots));
  cfg.blockDim = dim3(kFusedThreads, 1, 1);
  cfg.dynamicSmemBytes = fused_smem_bytes(a.dim);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeCooperative;   // the gate exchange needs co-residency
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, engram_fused_kernel, tmA, tmWk, tmWv, tmX, p);
}

}  // namespace engram
