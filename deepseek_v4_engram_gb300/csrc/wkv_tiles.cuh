// Tile geometry and pipeline helpers shared by the tensor-core kernels of the wkv projection.
#pragma once

#include "device.cuh"

namespace engram {

constexpr int kBM = 128;              // tokens per tile (MMA M)
constexpr int kBN = 256;              // kv columns per tile (MMA N)
constexpr int kBK = 64;               // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kUmmaK = 16;            // K of one tcgen05.mma kind::f16
constexpr int kStages = 4;            // shared-memory ring depth
constexpr int kTileABytes = kBM * kBK * 2;
constexpr int kTileBBytes = kBN * kBK * 2;
constexpr uint32_t kTmemCols = 512;   // two kBN-column f32 accumulators
constexpr int kEpilogueThreads = 128;

__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Wait for a phase with a time limit only (used while tearing down, when abort is already set).
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
  }
}

// Producer side of a ring of kSlots TMA buffers: which slot to fill next, and which loads are in
// flight so they can be waited for before the CTA exits.
template <int kSlots>
struct TmaRingT {
  uint32_t stage = 0, phase = 0;
  uint32_t issued_mask = 0;
  uint32_t issued_parity = 0;  // bit s: parity of the last load issued into stage s

  __device__ __forceinline__ bool acquire(uint64_t* empty, volatile int* abort, uint32_t* err) {
    return mbar_wait(&empty[stage], phase ^ 1u, abort, err);
  }
  __device__ __forceinline__ void issued() {
    issued_mask |= 1u << stage;
    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
    if (++stage == kSlots) {
      stage = 0;
      phase ^= 1u;
    }
  }
  // Wait (bounded) until every issued load has landed.
  __device__ __forceinline__ void drain(uint64_t* full) {
    for (int s = 0; s < kSlots; ++s)
      if (issued_mask & (1u << s)) mbar_wait_drain(&full[s], (issued_parity >> s) & 1u);
  }
};

using TmaRing = TmaRingT<kStages>;

}  // namespace engram
