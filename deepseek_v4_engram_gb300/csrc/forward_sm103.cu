// Stages 3 + 4 fused: the wkv projection on the tensor cores with the gate-and-add in its
// epilogue, so the dim * (hc + 1)-wide kv row never goes to HBM.
//
// Engram listing, forward: kv = wkv(rows); key, value = split(kv); per (token, stream) the three
// sums over dim (h^2, key^2, h*w*key) give the gate; out = bf16(h + gate * value).
//
// Work split: one thread-block cluster of hc CTAs per 128-token tile. CTA s of the cluster owns
// stream s: it computes the key columns [s*dim, (s+1)*dim) in 256-wide tiles and accumulates the
// sums of stream s for its 128 tokens entirely on its own (no cross-CTA reduction of partial
// sums). It then computes its share [s*dim/hc, (s+1)*dim/hc) of the value columns. Between the
// two phases the hc CTAs swap their 128 gates through distributed shared memory (one float per
// token per CTA, remote stores + remote mbarrier arrivals), so each CTA can write
// out[m, s', cols] = h + gate[m, s'] * value for all hc streams of its value columns.
//
// Roles per CTA (224 threads):
//   warp 0      TMA producer of the GEMM operands (A rows, wkv rows) into a 3-stage ring;
//   warp 1      TMEM owner + MMA issuer (two 256-column f32 accumulators);
//   warps 2-5   epilogue, thread = token row: tcgen05.ld of the accumulator, gate sums, output;
//   warp 6      TMA producer of the residual streams x: 128-token x 64-column boxes into a
//               4-slot ring, in exactly the order the epilogue consumes them, so the epilogue
//               never waits on a global-memory round trip for x.
#include "device.cuh"
#include "kernels.h"
#include "wkv_tiles.cuh"

namespace engram {

namespace {

constexpr int kFusedThreads = 224;
constexpr int kFusedStages = 3;            // A/B ring depth
constexpr int kXSlots = 4;                 // x ring depth
constexpr int kXCols = 64;                 // columns per x box (128 B per row: one swizzle row)
constexpr int kXBoxBytes = kBM * kXCols * 2;
constexpr int kMaxHc = 8;

struct FusedShared {
  uint64_t full[kFusedStages];
  uint64_t empty[kFusedStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t xfull[kXSlots];
  uint64_t xempty[kXSlots];
  uint64_t drain;
  uint64_t gate_bar;            // completes when every CTA of the cluster delivered its gates
  uint32_t tmem_base;
  int abort;
  float gates[kMaxHc][kBM];     // gates[s][row]: written by CTA s of the cluster
};

constexpr size_t kFusedSmem = size_t(kFusedStages) * (kTileABytes + kTileBBytes) +
                              size_t(kXSlots) * kXBoxBytes + sizeof(FusedShared) + 1024;

struct FusedParams {
  const uint16_t* q;
  const uint16_t* k;
  const uint8_t* mask;
  uint16_t* out;
  float* gate_out;
  uint16_t* kv_out;
  int64_t M;
  int32_t K, hc, dim, bnv;
  float eps, inv_sqrt_dim;
  uint32_t* err;
  LenAdvance adv;
};

// Value columns per CTA are split into tiles of bnv columns: the largest multiple of 64 that
// divides dim / hc and is at most 256.
int value_tile_width(int32_t hc, int32_t dim) {
  if (hc <= 0 || dim % hc != 0) return 0;
  const int v = dim / hc;
  for (int w = 256; w >= 64; w -= 64)
    if (v % w == 0) return w;
  return 0;
}

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void load_bf16x32_global(const uint16_t* p, uint32_t (&v)[16]) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 t = __ldg(q + i);
    v[4 * i + 0] = t.x;
    v[4 * i + 1] = t.y;
    v[4 * i + 2] = t.z;
    v[4 * i + 3] = t.w;
  }
}

template <int kWords>
__device__ __forceinline__ void store_words(uint16_t* p, const uint32_t* v) {
  uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int i = 0; i < kWords / 4; ++i)
    q[i] = make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

// One row (64 bf16 = 128 B) of a 128B-swizzled x box: 16-byte chunk j of row r sits at chunk
// position j ^ (r % 8).
__device__ __forceinline__ void read_x_row(const uint8_t* box, int row, uint32_t (&v)[32]) {
  const uint32_t base = smem_u32(box) + row * 128;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint4 t = lds128(base + ((j ^ (row & 7)) << 4));
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
    advance();
  }
  __device__ __forceinline__ void advance() {
    if (++slot == kXSlots) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

__global__ void __launch_bounds__(kFusedThreads, 1)
    engram_fused_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmWk,
                        const __grid_constant__ CUtensorMap tmWv,
                        const __grid_constant__ CUtensorMap tmX, const FusedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = sA + kFusedStages * kTileABytes;
  uint8_t* sX = sB + kFusedStages * kTileBBytes;
  FusedShared* sh = reinterpret_cast<FusedShared*>(sX + kXSlots * kXBoxBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t s = static_cast<int32_t>(cluster_ctarank());   // this CTA's stream
  const int32_t hc = p.hc, dim = p.dim, bnv = p.bnv;
  const int32_t m0 = static_cast<int32_t>(blockIdx.y) * kBM;
  const int32_t vcols = dim / hc;
  const int nk = dim / kBN;                 // key tiles
  const int nv = vcols / bnv;               // value tiles
  const int ntiles = nk + nv;
  const int kblocks = p.K / kBK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kFusedStages; ++i) {
      mbar_init(&sh->full[i], 1);
      mbar_init(&sh->empty[i], 1);
    }
    for (int i = 0; i < kXSlots; ++i) {
      mbar_init(&sh->xfull[i], 1);
      mbar_init(&sh->xempty[i], kEpilogueThreads);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->tfull[a], 1);
      mbar_init(&sh->tempty[a], kEpilogueThreads);
    }
    mbar_init(&sh->drain, 1);
    mbar_init(&sh->gate_bar, static_cast<uint32_t>(hc * kEpilogueThreads));
    sh->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmWk);
    tma_prefetch_desc(&tmWv);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(&sh->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync_all();   // barriers of every CTA initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;
  volatile int* abort = &sh->abort;
  pdl_wait();   // rows (and the cache lengths) come from the previous kernel of the stream
  pdl_launch_dependents();
  if (p.adv.len != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < 32)
    for (int32_t b = threadIdx.x; b < p.adv.B; b += 32)
      p.adv.len[b] = min(p.adv.len[b] + p.adv.T, p.adv.cap);

  if (warp == 0) {
    // ------------------------------------------------------------- GEMM operand producer
    if (lane == 0) {
      TmaRingT<kFusedStages> ring;
      for (int t = 0; t < ntiles && !*abort; ++t) {
        const bool key = t < nk;
        const int32_t n0 = key ? s * dim + t * kBN : hc * dim + s * vcols + (t - nk) * bnv;
        const uint32_t bbytes = static_cast<uint32_t>((key ? kBN : bnv) * kBK * 2);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ring.acquire(sh->empty, abort, p.err)) break;
          mbar_arrive_expect_tx(&sh->full[ring.stage], kTileABytes + bbytes);
          tma_load_2d(sA + ring.stage * kTileABytes, &tmA, &sh->full[ring.stage], kb * kBK, m0);
          tma_load_2d(sB + ring.stage * kTileBBytes, key ? &tmWk : &tmWv, &sh->full[ring.stage],
                      kb * kBK, n0);
          ring.issued();
        }
      }
      ring.drain(sh->full);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc_k = idesc_bf16_f32(kBM, kBN);
      const uint32_t idesc_v = idesc_bf16_f32(kBM, bnv);
      uint32_t stage = 0, phase = 0;
      for (int t = 0; t < ntiles && !*abort; ++t) {
        const uint32_t acc = t & 1, acc_phase = (t >> 1) & 1;
        if (!mbar_wait(&sh->tempty[acc], acc_phase ^ 1u, abort, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * kBN;
        const uint32_t idesc = t < nk ? idesc_k : idesc_v;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&sh->full[stage], phase, abort, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad = sw128_kmajor_desc(smem_u32(sA + stage * kTileABytes));
          const uint64_t bd = sw128_kmajor_desc(smem_u32(sB + stage * kTileBBytes));
#pragma unroll
          for (int kk = 0; kk < kBK / kUmmaK; ++kk)
            tc_mma_bf16(d, ad + 2ull * kk, bd + 2ull * kk, idesc, (kb | kk) != 0);
          tc_commit(&sh->empty[stage]);
          if (++stage == kFusedStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(&sh->tfull[acc]);
      }
      tc_commit(&sh->drain);
      mbar_wait_drain(&sh->drain, 0);
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------- x producer
    // Same order as the epilogue: key tiles (stream s, 4 boxes each), then value tiles (for each
    // 64-column box of the tile, the hc streams in turn).
    if (lane == 0) {
      TmaRingT<kXSlots> ring;
      const int total_steps = nk * (kBN / kXCols) + nv * (bnv / kXCols) * hc;
      for (int q = 0; q < total_steps && !*abort; ++q) {
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
        tma_load_3d(sX + ring.stage * kXBoxBytes, &tmX, &sh->xfull[ring.stage], col, stream, m0);
        ring.issued();
      }
      ring.drain(sh->xfull);
    }
  } else {
    // ------------------------------------------------------------- epilogue (warps 2-5)
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const int64_t m = static_cast<int64_t>(m0) + row;
    const bool valid = m < p.M;
    const bool keep = valid && (p.mask == nullptr || p.mask[m] != 0);
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const int64_t N = static_cast<int64_t>(dim) * (hc + 1);
    float sh2 = 0.f, sk2 = 0.f, shwk = 0.f;
    float gl[kMaxHc];
#pragma unroll
    for (int i = 0; i < kMaxHc; ++i) gl[i] = 0.f;
    XRing xr;

    for (int t = 0; t < ntiles; ++t) {
      const uint32_t acc = t & 1, acc_phase = (t >> 1) & 1;
      if (!mbar_wait(&sh->tfull[acc], acc_phase, abort, p.err)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + lane_base + acc * kBN;
      bool ok = true;
      if (t < nk) {
        // key tile: columns d0 .. d0 + 255 of stream s, in four 64-column boxes
        const int32_t d0 = t * kBN;
        for (int c4 = 0; c4 < kBN / kXCols && ok; ++c4) {
          if (!mbar_wait(&sh->xfull[xr.slot], xr.phase, abort, p.err)) { ok = false; break; }
          uint32_t xv[32];
          read_x_row(sX + xr.slot * kXBoxBytes, row, xv);
          xr.release(sh->xempty);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t r[32];
            tc_ld_32x32b_x32(tbase + c4 * kXCols + half * 32, r);
            const int32_t d = d0 + c4 * kXCols + half * 32;
            uint32_t qv[16], kv[16], kb16[16];
            load_bf16x32_global(p.q + static_cast<int64_t>(s) * dim + d, qv);
            load_bf16x32_global(p.k + static_cast<int64_t>(s) * dim + d, kv);
            tc_wait_ld(r);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              kb16[e] = pack_bf16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]));
              const uint32_t xw = xv[half * 16 + e];
              const float key0 = lo_bf16(kb16[e]), key1 = hi_bf16(kb16[e]);
              const float h0 = lo_bf16(xw), h1 = hi_bf16(xw);
              const float w0 = lo_bf16(qv[e]) * lo_bf16(kv[e]);
              const float w1 = hi_bf16(qv[e]) * hi_bf16(kv[e]);
              sh2 = fmaf(h0, h0, sh2);
              sk2 = fmaf(key0, key0, sk2);
              shwk = fmaf(h0 * w0, key0, shwk);
              sh2 = fmaf(h1, h1, sh2);
              sk2 = fmaf(key1, key1, sk2);
              shwk = fmaf(h1 * w1, key1, shwk);
            }
            if (valid && p.kv_out)
              store_words<16>(p.kv_out + m * N + static_cast<int64_t>(s) * dim + d, kb16);
          }
        }
      } else {
        // value tile: value columns col0 .. col0 + bnv - 1, shared by all hc streams
        const int32_t col0 = s * vcols + (t - nk) * bnv;
        for (int c4 = 0; c4 < bnv / kXCols && ok; ++c4) {
          const int32_t col = col0 + c4 * kXCols;
          uint32_t vb[32];
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t r[32];
            tc_ld_32x32b_x32(tbase + c4 * kXCols + half * 32, r);
            tc_wait_ld(r);
#pragma unroll
            for (int e = 0; e < 16; ++e)
              vb[half * 16 + e] = pack_bf16x2(__uint_as_float(r[2 * e]),
                                              __uint_as_float(r[2 * e + 1]));
          }
          if (valid && p.kv_out)
            store_words<32>(p.kv_out + m * N + static_cast<int64_t>(hc) * dim + col, vb);
          for (int s2 = 0; s2 < hc; ++s2) {
            if (!mbar_wait(&sh->xfull[xr.slot], xr.phase, abort, p.err)) { ok = false; break; }
            uint32_t xv[32];
            read_x_row(sX + xr.slot * kXBoxBytes, row, xv);
            xr.release(sh->xempty);
            if (!valid) continue;
            if (keep) {
              float g = gl[0];
#pragma unroll
              for (int i = 1; i < kMaxHc; ++i) g = (s2 == i) ? gl[i] : g;
#pragma unroll
              for (int e = 0; e < 32; ++e)
                xv[e] = pack_bf16x2(fmaf(g, lo_bf16(vb[e]), lo_bf16(xv[e])),
                                    fmaf(g, hi_bf16(vb[e]), hi_bf16(xv[e])));
            }   // a masked token's x passes through unchanged
            store_words<32>(p.out + (m * hc + s2) * dim + col, xv);
          }
        }
      }
      if (!ok) break;
      tc_fence_before();
      mbar_arrive(&sh->tempty[acc]);

      if (t == nk - 1) {
        // all key tiles done: this CTA's gate for its 128 tokens, then swap gates with the
        // other CTAs of the cluster
        float g = 0.f;
        if (keep) g = gate_from_sums(sh2, sk2, shwk, dim, p.eps, p.inv_sqrt_dim);
        if (valid && p.gate_out) p.gate_out[m * hc + s] = g;
        const uint32_t slot = smem_u32(&sh->gates[s][row]);
        const uint32_t bar = smem_u32(&sh->gate_bar);
        for (int j = 0; j < hc; ++j) {
          st_cluster_f32(map_to_rank(slot, j), g);
          mbar_arrive_remote(map_to_rank(bar, j));
        }
        if (!mbar_wait<true>(&sh->gate_bar, 0, abort, p.err)) break;
#pragma unroll
        for (int i = 0; i < kMaxHc; ++i) gl[i] = i < hc ? sh->gates[i][row] : 0.f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

bool fused_supported(int32_t K, int32_t hc, int32_t dim) {
  return K > 0 && K % kBK == 0 && hc >= 1 && hc <= kMaxHc && dim % kBN == 0 &&
         value_tile_width(hc, dim) > 0;
}

cudaError_t launch_fused(const FusedArgs& a, cudaStream_t st, bool pdl) {
  const int bnv = value_tile_width(a.hc, a.dim);
  const int64_t N = static_cast<int64_t>(a.dim) * (a.hc + 1);
  alignas(64) CUtensorMap tmA, tmWk, tmWv, tmX;
  if (!tensor_map_2d_bf16(&tmA, a.a, a.K, a.M, kBK, kBM) ||
      !tensor_map_2d_bf16(&tmWk, a.w, a.K, N, kBK, kBN) ||
      !tensor_map_2d_bf16(&tmWv, a.w, a.K, N, kBK, bnv) ||
      !tensor_map_3d_bf16(&tmX, a.x, a.dim, a.hc, a.M, kXCols, 1, kBM))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(engram_fused_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kFusedSmem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  FusedParams p{};
  p.q = a.q;
  p.k = a.k;
  p.mask = a.mask;
  p.out = a.out;
  p.gate_out = a.gate_out;
  p.kv_out = a.kv_out;
  p.M = a.M;
  p.K = a.K;
  p.hc = a.hc;
  p.dim = a.dim;
  p.bnv = bnv;
  p.eps = a.eps;
  p.inv_sqrt_dim = a.inv_sqrt_dim;
  p.err = a.err;
  p.adv = a.adv;

  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(a.hc), static_cast<unsigned>((a.M + kBM - 1) / kBM), 1);
  cfg.blockDim = dim3(kFusedThreads, 1, 1);
  cfg.dynamicSmemBytes = kFusedSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(a.hc);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, engram_fused_kernel, tmA, tmWk, tmWv, tmX, p);
}

}  // namespace engram
