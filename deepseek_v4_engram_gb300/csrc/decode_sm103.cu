// Stage 3 for decode-sized batches (M <= 64 tokens): the wkv projection as a weight-streaming
// tensor-core GEMM that reads the 78.6 MB weight once, spread evenly over every SM, and writes
// bf16 kv (3.3 MB at 64 tokens) for the gate kernel.
//
// Page "Module engram", stage 3 / linear_bf16: kv = a @ w^T, bf16 in, f32 accumulate, bf16 out.
// The weight is cut into units of 64 rows (400 at full width); CTA i owns units i, i + grid,
// i + 2 * grid (at most three), so every SM streams nearly the same share and no partial sums
// are needed. One K-loop per CTA covers all of its units: a ring stage holds one 64-row weight box
// per unit and one box of the activations, loaded once for every unit of the stage. Two units
// share one tcgen05 MMA (kind::f16, M = 128: unit a in rows 0-63, unit b in rows 64-127; N = the
// tokens rounded up to 32); a third unit's MMA has the activation box in rows 64-127, whose
// products are never read.
//
// Launched with programmatic dependent launch after the kernel that gathers the activations:
// the CTA requests the first K-blocks of its weight before it waits for that kernel, so the
// weight stream starts while the hash and gather still run.
//
// Roles per CTA (192 threads): warp 0 TMA producer; warp 1 TMEM owner and MMA issuer; warps 2-5
// epilogue (warp w reads TMEM lane quadrant w % 4 and stores its rows of kv, lane = kv column).
#include "device.cuh"
#include "kernels.h"
#include "wkv_tiles.cuh"

namespace engram {

namespace {

constexpr int kDecThreads = 192;
constexpr int kDecRows = 64;                      // wkv rows per unit
constexpr int kDecMaxTokens = 64;
constexpr int kDecMaxUnits = 3;                   // units per CTA
constexpr int kDecBoxBytes = kDecRows * kBK * 2;  // 8 KB: one weight box or the activation box
constexpr int kDecStageBytes = (kDecMaxUnits + 1) * kDecBoxBytes;   // 32 KB
constexpr int kDecStages = 6;
constexpr uint32_t kDecTmemCols = 128;            // two accumulators (unit pairs) of <= 64 columns

struct DecShared {
  uint64_t full[kDecStages];
  uint64_t empty[kDecStages];
  uint64_t tfull;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

size_t decode_smem_bytes() {
  return size_t(kDecStages) * kDecStageBytes + sizeof(DecShared) + 1024;
}

struct DecParams {
  uint16_t* kv;     // [M, N] bf16
  int32_t M, N, K, nt;
  uint32_t* err;
};

__global__ void __launch_bounds__(kDecThreads, 1)
    wkv_decode_kernel(const __grid_constant__ CUtensorMap tmW,
                      const __grid_constant__ CUtensorMap tmA, const DecParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  DecShared* sh = reinterpret_cast<DecShared*>(smem + kDecStages * kDecStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kblocks = p.K / kBK;
  const int32_t units_total = p.N / kDecRows;
  int32_t units[kDecMaxUnits];
  int nu = 0;
  for (int32_t u = blockIdx.x; u < units_total && nu < kDecMaxUnits; u += gridDim.x)
    units[nu++] = u;
  const int npairs = (nu + 1) / 2;
  const uint32_t tok_off = static_cast<uint32_t>(kDecMaxUnits) * kDecBoxBytes;   // activation box
  const uint32_t stage_tx = static_cast<uint32_t>(nu) * kDecBoxBytes +
                            static_cast<uint32_t>(p.nt) * kBK * 2;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kDecStages; ++i) {
      mbar_init(&sh->full[i], 1);
      mbar_init(&sh->empty[i], 1);
    }
    mbar_init(&sh->tfull, 1);
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmA);
  }
  if (warp == 1) {
    tmem_alloc(&sh->tmem_base, kDecTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;
  volatile int* abort = &sh->abort;

  if (warp == 0) {
    // ------------------------------------------------------------- TMA producer
    if (lane == 0) {
      // The weight is read once: its lines are the first to go when L2 needs room, so that the
      // stream replaces its own lines rather than evicting (and writing back) what earlier
      // kernels left there (measured: decode step 34.3 -> 32.0 us after a 256 MB write).
      const uint64_t stream_l2 = l2_evict_first_policy();
      // the weight does not depend on the previous kernel: its first K-blocks are requested
      // before waiting for it
      const int pre = nu == 0 ? 0 : (kblocks < kDecStages ? kblocks : kDecStages);
      for (int j = 0; j < pre; ++j) {
        mbar_arrive_expect_tx(&sh->full[j], stage_tx);
        for (int i = 0; i < nu; ++i)
          tma_load_2d_hint(smem + j * kDecStageBytes + i * kDecBoxBytes, &tmW, &sh->full[j],
                           j * kBK, units[i] * kDecRows, stream_l2);
      }
      pdl_wait();   // the activations come from the previous kernel of the stream
      pdl_launch_dependents();
      for (int j = 0; j < pre; ++j)
        tma_load_2d(smem + j * kDecStageBytes + tok_off, &tmA, &sh->full[j], j * kBK, 0);
      uint32_t stage = pre % kDecStages, phase = pre == kDecStages ? 1u : 0u;
      int issued = pre;   // K-blocks whose loads were issued
      for (int kb = pre; kb < kblocks && nu > 0; ++kb, ++issued) {
        uint8_t* st = smem + stage * kDecStageBytes;
        if (!mbar_wait(&sh->empty[stage], phase ^ 1u, abort, p.err)) break;
        mbar_arrive_expect_tx(&sh->full[stage], stage_tx);
        for (int i = 0; i < nu; ++i)
          tma_load_2d_hint(st + i * kDecBoxBytes, &tmW, &sh->full[stage], kb * kBK,
                           units[i] * kDecRows, stream_l2);
        tma_load_2d(st + tok_off, &tmA, &sh->full[stage], kb * kBK, 0);
        if (++stage == kDecStages) { stage = 0; phase ^= 1u; }
      }
      // every load issued has landed (each stage's last fill) before the CTA may exit
      for (int j = 0; j < kDecStages && j < issued; ++j) {
        const int last = ((issued - 1 - j) / kDecStages) * kDecStages + j;   // last fill of j
        mbar_wait_drain(&sh->full[j], static_cast<uint32_t>(last / kDecStages) & 1u);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0 && nu > 0) {
      const uint32_t idesc = idesc_bf16_f32(128, p.nt);
      uint32_t st = 0, ph = 0;
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!mbar_wait(&sh->full[st], ph, abort, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint8_t* sp = smem + st * kDecStageBytes;
        const uint64_t bd = sw128_kmajor_desc(smem_u32(sp + tok_off));
        for (int pr = 0; pr < npairs; ++pr) {
          // A: 128 rows from weight box 2 * pr (two units, or one unit and rows never read)
          const uint64_t ad = sw128_kmajor_desc(smem_u32(sp + 2 * pr * kDecBoxBytes));
          const uint32_t d = tmem_base + pr * (kDecTmemCols / 2);
#pragma unroll
          for (int kk = 0; kk < kBK / kUmmaK; ++kk)
            tc_mma_bf16(d, ad + 2ull * kk, bd + 2ull * kk, idesc, (kb | kk) != 0);
        }
        tc_commit(&sh->empty[st]);
        if (++st == kDecStages) { st = 0; ph ^= 1u; }
      }
      if (ok) tc_commit(&sh->tfull);
      tc_commit(&sh->drain);
      mbar_wait_drain(&sh->drain, 0);
    }
  } else {
    // ------------------------------------------------------------- epilogue (warps 2-5)
    const int quad = warp & 3;   // TMEM lane quadrant: 0-1 the first unit of a pair, 2-3 the second
    bool ok = nu > 0 && mbar_wait(&sh->tfull, 0, abort, p.err);
    ok = __all_sync(0xFFFFFFFFu, ok);
    if (ok) {
      tc_fence_after();
      for (int pr = 0; pr < npairs; ++pr) {
        const int ui = 2 * pr + (quad >> 1);
        if (ui >= nu) continue;
        const int64_t n = static_cast<int64_t>(units[ui]) * kDecRows + (quad & 1) * 32 + lane;
        for (int c = 0; c < p.nt / 32; ++c) {
          uint32_t r[32];
          tc_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                               pr * (kDecTmemCols / 2) + c * 32,
                           r);
          tc_wait_ld(r);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int m = c * 32 + j;
            if (m < p.M)   // consecutive lanes write consecutive columns of token m
              p.kv[static_cast<int64_t>(m) * p.N + n] =
                  static_cast<uint16_t>(pack_bf16x2(__uint_as_float(r[j]), 0.f));
          }
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
    tmem_dealloc(tmem_base, kDecTmemCols);
  }
}

int dec_sm_count() { return device_sm_count(); }

}  // namespace

bool decode_supported(int64_t M, int32_t N, int32_t K) {
  return M >= 1 && M <= kDecMaxTokens && K % kBK == 0 && N % kDecRows == 0 &&
         N / kDecRows <= kDecMaxUnits * dec_sm_count();
}

cudaError_t launch_wkv_decode(const WkvSmallArgs& a, cudaStream_t st, bool pdl) {
  const int32_t M = static_cast<int32_t>(a.M);
  const int32_t nt = (M + 31) / 32 * 32;
  const int32_t units = a.N / kDecRows;
  const int32_t grid = units < dec_sm_count() ? units : dec_sm_count();
  alignas(64) CUtensorMap tmW, tmA;
  if (!tensor_map_2d_bf16(&tmW, a.w, a.K, a.N, kBK, kDecRows) ||
      !tensor_map_2d_bf16(&tmA, a.a, a.K, M, kBK, nt))
    return cudaErrorInvalidValue;
  const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(wkv_decode_kernel),
                                            decode_smem_bytes());
  if (e != cudaSuccess) return e;
  DecParams p{};
  p.kv = a.kv;
  p.M = M;
  p.N = a.N;
  p.K = a.K;
  p.nt = nt;
  p.err = a.err;
  return launch_ex(wkv_decode_kernel, dim3(static_cast<unsigned>(grid)), dim3(kDecThreads),
                   decode_smem_bytes(), st, pdl, tmW, tmA, p);
}

}  // namespace engram
