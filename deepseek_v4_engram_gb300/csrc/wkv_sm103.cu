// Stage 3, the wkv projection, on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
// Page "Module engram", stage 3 / linear_bf16: kv = a @ w^T, bf16 in, f32 accumulate, bf16 out.
//
// Persistent, warp-specialised kernel, one CTA per SM:
//   warp 0      TMA producer: A tile [128 x 64] and W tile [BN x 64] per K-block into a ring of
//               shared-memory stages (128-byte swizzle), completion on a "full" mbarrier;
//   warp 1      owns TMEM (512 columns = two BN=256 f32 accumulators) and issues tcgen05.mma
//               (M=128, N=BN, K=16) from one thread; tcgen05.commit frees each stage and, after
//               the last K-block, marks the accumulator full;
//   warps 2-5   epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes 32*(w%4)...),
//               round to bf16, store, release the accumulator to the MMA warp.
// Two accumulators let the epilogue of tile i overlap the main loop of tile i+1.
#include <cstdio>

#include "device.cuh"
#include "kernels.h"
#include "wkv_tiles.cuh"

namespace engram {

namespace {

constexpr int kGemmThreads = 192;

struct GemmShared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

__global__ void __launch_bounds__(kGemmThreads, 1)
    wkv_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    uint16_t* __restrict__ kv, int64_t M, int32_t N, int32_t K, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint8_t* sA = smem;                                   // kStages x 16 KB
  uint8_t* sB = smem + kStages * kTileABytes;           // kStages x 32 KB
  GemmShared* sh = reinterpret_cast<GemmShared*>(sB + kStages * kTileBBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t num_m = (M + kBM - 1) / kBM;
  const int64_t num_n = (N + kBN - 1) / kBN;
  const int64_t tiles = num_m * num_n;
  const int kblocks = K / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh->full[s], 1);
      mbar_init(&sh->empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->tfull[a], 1);
      mbar_init(&sh->tempty[a], kEpilogueThreads);
    }
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&sh->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;
  volatile int* abort = &sh->abort;
  // L2 policies: with few M tiles (up to 8: 1024 tokens), a weight tile serves the M tiles that
  // run at the same time and is then done with (evict-first; measured 3.5-4 us faster at 384 and
  // 1024 tokens); with more, its readers are spread out in time and it keeps the default policy
  // (evict-first there cost 3% at 4096). The activations serve every N tile (evict-last).
  const bool stream_w = num_m <= 8;
  const uint64_t once = l2_evict_first_policy(), keep = l2_evict_last_policy();
  // The weight does not depend on the previous kernel: the first tile's first stages of it are
  // requested before waiting for that kernel (with the policies above: the forward at 384 tokens
  // 57.1 -> 53.0 us).
  int pre = 0;
  if (warp == 0 && lane == 0 && static_cast<int64_t>(blockIdx.x) < tiles) {
    const int32_t n0 = static_cast<int32_t>((blockIdx.x / num_m) * kBN);
    pre = kblocks < kStages ? kblocks : kStages;
    for (int kb = 0; kb < pre; ++kb) {   // a fresh ring: stage kb is free
      mbar_arrive_expect_tx(&sh->full[kb], kTileABytes + kTileBBytes);
      if (stream_w)
        tma_load_2d_hint(sB + kb * kTileBBytes, &tmB, &sh->full[kb], kb * kBK, n0, once);
      else
        tma_load_2d(sB + kb * kTileBBytes, &tmB, &sh->full[kb], kb * kBK, n0);
    }
  }
  pdl_wait();   // the activations come from the previous kernel of the stream
  pdl_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      TmaRing ring;
      for (int64_t tile = blockIdx.x; tile < tiles && !*abort; tile += gridDim.x) {
        const int32_t m0 = static_cast<int32_t>((tile % num_m) * kBM);
        const int32_t n0 = static_cast<int32_t>((tile / num_m) * kBN);
        for (int kb = 0; kb < kblocks; ++kb) {
          const bool preissued = tile == static_cast<int64_t>(blockIdx.x) && kb < pre;
          if (!preissued) {
            if (!ring.acquire(sh->empty, abort, err)) break;
            mbar_arrive_expect_tx(&sh->full[ring.stage], kTileABytes + kTileBBytes);
            if (stream_w)
              tma_load_2d_hint(sB + ring.stage * kTileBBytes, &tmB, &sh->full[ring.stage],
                               kb * kBK, n0, once);
            else
              tma_load_2d(sB + ring.stage * kTileBBytes, &tmB, &sh->full[ring.stage], kb * kBK,
                          n0);
          }
          tma_load_2d_hint(sA + ring.stage * kTileABytes, &tmA, &sh->full[ring.stage], kb * kBK,
                           m0, keep);
          ring.issued();
        }
      }
      ring.drain(sh->full);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kBM, kBN);
      uint32_t stage = 0, phase = 0;
      int64_t local = 0;
      for (int64_t tile = blockIdx.x; tile < tiles && !*abort; tile += gridDim.x, ++local) {
        const uint32_t acc = static_cast<uint32_t>(local & 1);
        const uint32_t acc_phase = static_cast<uint32_t>((local >> 1) & 1);
        if (!mbar_wait(&sh->tempty[acc], acc_phase ^ 1u, abort, err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * kBN;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&sh->full[stage], phase, abort, err)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad = sw128_kmajor_desc(smem_u32(sA + stage * kTileABytes));
          const uint64_t bd = sw128_kmajor_desc(smem_u32(sB + stage * kTileBBytes));
#pragma unroll
          for (int kk = 0; kk < kBK / kUmmaK; ++kk)
            tc_mma_bf16(d, ad + 2ull * kk, bd + 2ull * kk, idesc, (kb | kk) != 0);
          tc_commit(&sh->empty[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(&sh->tfull[acc]);
      }
      // Every MMA this thread issued has finished before TMEM is released.
      tc_commit(&sh->drain);
      mbar_wait_drain(&sh->drain, 0);
    }
  } else {
    const int quad = warp & 3;                    // TMEM lanes this warp may read
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    int64_t local = 0;
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++local) {
      const uint32_t acc = static_cast<uint32_t>(local & 1);
      const uint32_t acc_phase = static_cast<uint32_t>((local >> 1) & 1);
      if (!mbar_wait(&sh->tfull[acc], acc_phase, abort, err)) break;
      tc_fence_after();
      const int64_t m = (tile % num_m) * kBM + quad * 32 + lane;
      const int32_t n0 = static_cast<int32_t>((tile / num_m) * kBN);
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t r[32];
        tc_ld_32x32b_x32(tmem_base + lane_base + acc * kBN + c * 32, r);
        tc_wait_ld(r);
        if (m < M && n0 + c * 32 < N) {
          uint4* dst = reinterpret_cast<uint4*>(kv + m * N + n0 + c * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            dst[v] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * v + 0]), __uint_as_float(r[8 * v + 1])),
                                pack_bf16x2(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3])),
                                pack_bf16x2(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5])),
                                pack_bf16x2(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7])));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&sh->tempty[acc]);
    }
  }

  tc_fence_before();
  __syncwarp();
  cta_sync_all();   // every role is done with TMEM (each thread counted on its own)
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

int num_sms() { return device_sm_count(); }

}  // namespace

cudaError_t launch_wkv(const WkvArgs& a, cudaStream_t st, bool pdl) {
  alignas(64) CUtensorMap tmA, tmB;
  if (!tensor_map_2d_bf16(&tmA, a.a, a.K, a.M, kBK, kBM)) return cudaErrorInvalidValue;
  if (!tensor_map_2d_bf16(&tmB, a.w, a.K, a.N, kBK, kBN)) return cudaErrorInvalidValue;
  const size_t smem = kStages * (kTileABytes + kTileBBytes) + sizeof(GemmShared) + 1024;
  {
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(wkv_gemm_kernel), smem);
    if (e != cudaSuccess) return e;
  }
  const int64_t tiles = ((a.M + kBM - 1) / kBM) * ((a.N + kBN - 1) / kBN);
  const int grid = static_cast<int>(tiles < num_sms() ? tiles : num_sms());
  return launch_ex(wkv_gemm_kernel, dim3(grid), dim3(kGemmThreads), smem, st, pdl, tmA, tmB, a.kv,
                   a.M, a.N, a.K, a.err);
}

}  // namespace engram
