// Stage 3 for few tokens (decode): the wkv projection as a weight-streaming tensor-core GEMM.
// Page "Module engram", stage 3 / linear_bf16: kv = a @ w^T, bf16 in, f32 accumulate.
//
// With M <= 256 tokens the 78.6 MB weight dominates: the kernel must stream it once, at HBM
// bandwidth, over every SM. So the roles of the operands are swapped: a 128-row slice of wkv is
// the MMA's M side (tcgen05.mma M = 128) and the tokens are its N side (N = M rounded up to 16):
//   D[n, m] (+)= sum_k W[n, k] * a[m, k]   (D: 128 wkv rows x Nt tokens, in TMEM)
// Work items are (128-row slice, K part); K is split so that the items cover the SMs evenly
// (200 slices x 3 parts on 152 SMs at full width). A persistent CTA per SM walks its items
// through a deep TMA ring (W box 128 x 64, activation box Nt x 64, 128-byte swizzle).
//
// Output: with one K part the epilogue rounds to bf16 and writes kv[m, n]; with several it
// writes f32 partial sums part[kp, m, n], which the gate kernel adds in K order before rounding.
// Stores are coalesced across the warp (lane = wkv row n).
#include "device.cuh"
#include "kernels.h"
#include "wkv_tiles.cuh"

namespace engram {

namespace {

constexpr int kSmallThreads = 192;
constexpr int kSmallBM = 128;                 // wkv rows per item (MMA M)
constexpr int kSmallMaxN = 256;               // tokens per MMA (MMA N)
constexpr int kSmallMaxStages = 8;
constexpr int kSmallSmemBudget = 200 * 1024;  // operand ring

struct SmallShared {
  uint64_t full[kSmallMaxStages];
  uint64_t empty[kSmallMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

struct SmallParams {
  uint16_t* kv;        // [M, N] bf16 (ksplit == 1)
  float* part;         // [ksplit, M, N] f32 (ksplit > 1)
  int64_t M;
  int32_t N, K, nt, ksplit, stages;
  uint32_t* err;
};

__global__ void __launch_bounds__(kSmallThreads, 1)
    wkv_small_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                     const SmallParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  const int S = p.stages;
  const int a_bytes = kSmallBM * kBK * 2;                 // W slice box (MMA A operand)
  const int b_bytes = p.nt * kBK * 2;                     // token box (MMA B operand)
  const int stage_bytes = (a_bytes + b_bytes + 1023) & ~1023;
  SmallShared* sh = reinterpret_cast<SmallShared*>(smem + S * stage_bytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_slices = p.N / kSmallBM;
  const int items = n_slices * p.ksplit;
  const int kb_per = p.K / kBK / p.ksplit;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&sh->full[i], 1);
      mbar_init(&sh->empty[i], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sh->tfull[a], 1);
      mbar_init(&sh->tempty[a], kEpilogueThreads);
    }
    mbar_init(&sh->drain, 1);
    sh->abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmA);
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

  if (warp == 0) {
    if (lane == 0) {
      // producer: a ring of S stages. The wkv slices do not depend on earlier kernels, so the
      // first stages' weight loads are issued before waiting for the kernel that wrote the
      // activations (with a programmatic launch that wait overlaps the previous kernel's tail).
      // the weight is read once: evict-first, so that it replaces its own lines in L2
      const uint64_t stream_l2 = l2_evict_first_policy();
      uint32_t stage = 0, phase = 0, issued_mask = 0, issued_parity = 0;
      int pre = 0;
      if (static_cast<int>(blockIdx.x) < items) {
        const int n0 = (blockIdx.x / p.ksplit) * kSmallBM;
        const int kb0 = (blockIdx.x % p.ksplit) * kb_per;
        pre = kb_per < S ? kb_per : S;
        for (int j = 0; j < pre; ++j) {
          mbar_arrive_expect_tx(&sh->full[j], a_bytes + b_bytes);
          tma_load_2d_hint(smem + j * stage_bytes, &tmW, &sh->full[j], (kb0 + j) * kBK, n0,
                           stream_l2);
        }
      }
      pdl_wait();
      pdl_launch_dependents();
      bool ok = true;
      int g = 0;   // kblocks issued by this CTA so far
      for (int it = blockIdx.x; it < items && ok && !*abort; it += gridDim.x) {
        const int n0 = (it / p.ksplit) * kSmallBM;
        const int kb0 = (it % p.ksplit) * kb_per;
        for (int kb = kb0; kb < kb0 + kb_per; ++kb, ++g) {
          uint8_t* st = smem + stage * stage_bytes;
          if (g >= pre) {
            if (!mbar_wait(&sh->empty[stage], phase ^ 1u, abort, p.err)) { ok = false; break; }
            mbar_arrive_expect_tx(&sh->full[stage], a_bytes + b_bytes);
            tma_load_2d_hint(st, &tmW, &sh->full[stage], kb * kBK, n0, stream_l2);
          }
          tma_load_2d(st + a_bytes, &tmA, &sh->full[stage], kb * kBK, 0);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == static_cast<uint32_t>(S)) { stage = 0; phase ^= 1u; }
        }
      }
      for (int s2 = 0; s2 < S; ++s2)
        if (issued_mask & (1u << s2)) mbar_wait_drain(&sh->full[s2], (issued_parity >> s2) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kSmallBM, p.nt);
      uint32_t stage = 0, phase = 0;
      int local = 0;
      for (int it = blockIdx.x; it < items && !*abort; it += gridDim.x, ++local) {
        const uint32_t acc = local & 1, acc_phase = (local >> 1) & 1;
        if (!mbar_wait(&sh->tempty[acc], acc_phase ^ 1u, abort, p.err)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * kSmallMaxN;
        bool ok = true;
        for (int j = 0; j < kb_per; ++j) {
          if (!mbar_wait(&sh->full[stage], phase, abort, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint8_t* st = smem + stage * stage_bytes;
          const uint64_t ad = sw128_kmajor_desc(smem_u32(st));
          const uint64_t bd = sw128_kmajor_desc(smem_u32(st + a_bytes));
#pragma unroll
          for (int kk = 0; kk < kBK / kUmmaK; ++kk)
            tc_mma_bf16(d, ad + 2ull * kk, bd + 2ull * kk, idesc, (j | kk) != 0);
          tc_commit(&sh->empty[stage]);
          if (++stage == static_cast<uint32_t>(S)) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        tc_commit(&sh->tfull[acc]);
      }
      tc_commit(&sh->drain);
      mbar_wait_drain(&sh->drain, 0);
    }
  } else {
    const int quad = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    int local = 0;
    for (int it = blockIdx.x; it < items; it += gridDim.x, ++local) {
      const uint32_t acc = local & 1, acc_phase = (local >> 1) & 1;
      if (!mbar_wait(&sh->tfull[acc], acc_phase, abort, p.err)) break;
      tc_fence_after();
      const int64_t n = static_cast<int64_t>(it / p.ksplit) * kSmallBM + quad * 32 + lane;
      const int kp = it % p.ksplit;
#pragma unroll 1
      for (int c = 0; c < p.nt / 32; ++c) {
        uint32_t r[32];
        tc_ld_32x32b_x32(tmem_base + lane_base + acc * kSmallMaxN + c * 32, r);
        tc_wait_ld(r);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int64_t m = c * 32 + j;
          if (m < p.M) {
            if (p.ksplit == 1)
              p.kv[m * p.N + n] = static_cast<uint16_t>(pack_bf16x2(__uint_as_float(r[j]), 0.f));
            else
              p.part[(kp * p.M + m) * p.N + n] = __uint_as_float(r[j]);
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

int sm_count() { return device_sm_count(); }

}  // namespace

bool small_supported(int64_t M, int32_t N, int32_t K) {
  return M >= 1 && M <= kSmallMaxN && N % kSmallBM == 0 && K % kBK == 0;
}

// K parts for the weight-streaming GEMM: the divisor of K / 64 that brings the item count
// closest to (without exceeding much) a whole number of passes over the SMs.
int small_ksplit(int32_t N, int32_t K) {
  const int slices = N / kSmallBM, kblocks = K / kBK, sms = sm_count();
  int best = 1;
  double best_eff = 0.0;
  for (int ks = 1; ks <= 8; ++ks) {
    if (kblocks % ks != 0) continue;
    const int items = slices * ks;
    const int passes = (items + sms - 1) / sms;
    const double eff = double(items) / double(passes * sms);   // SM balance
    if (eff > best_eff + 0.02) {
      best_eff = eff;
      best = ks;
    }
  }
  return best;
}

cudaError_t launch_wkv_small(const WkvSmallArgs& a, cudaStream_t st, bool pdl) {
  const int nt = static_cast<int>((a.M + 31) / 32 * 32);   // tokens per MMA, a multiple of 32
  alignas(64) CUtensorMap tmW, tmA;
  if (!tensor_map_2d_bf16(&tmW, a.w, a.K, a.N, kBK, kSmallBM) ||
      !tensor_map_2d_bf16(&tmA, a.a, a.K, a.M, kBK, nt))
    return cudaErrorInvalidValue;
  const int stage_bytes = ((kSmallBM + nt) * kBK * 2 + 1023) & ~1023;
  int stages = kSmallSmemBudget / stage_bytes;
  if (stages > kSmallMaxStages) stages = kSmallMaxStages;
  const size_t smem = size_t(stages) * stage_bytes + sizeof(SmallShared) + 1024;
  {
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(wkv_small_kernel),
                                              kSmallSmemBudget + sizeof(SmallShared) + 2048);
    if (e != cudaSuccess) return e;
  }
  SmallParams p{};
  p.kv = a.kv;
  p.part = a.part;
  p.M = a.M;
  p.N = a.N;
  p.K = a.K;
  p.nt = nt;
  p.ksplit = a.ksplit;
  p.stages = stages;
  p.err = a.err;
  const int items = (a.N / kSmallBM) * a.ksplit;
  const int grid = items < sm_count() ? items : sm_count();
  return launch_ex(wkv_small_kernel, dim3(grid), dim3(kSmallThreads), smem, st, pdl, tmW, tmA, p);
}

}  // namespace engram
