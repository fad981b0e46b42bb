// A measurement kernel, not a stage of the forward: one read of a device buffer spread over every
// SM, with nothing done with the bytes. It bounds from below what a kernel that streams the same
// buffer once (the decode projection streaming the wkv weight) can take in the same memory state,
// whatever it computes.
//
// Each CTA (one per SM) reads a contiguous share of the buffer, either
//  - kBulk: as 32 KB bulk copies (cp.async.bulk) into a 6-stage shared-memory ring, one thread
//    issuing, 192 KB in flight per SM as in the decode projection's ring; or
//  - kPlain: as 16-byte non-caching loads by 512 threads, four per thread in flight, XOR-folded
//    into one word per CTA so that the loads cannot be dropped;
//  - kBulkEvictFirst: as kBulk, with an L2 evict-first policy on the copies (what the decode
//    projection uses for the weight).
#include "device.cuh"
#include "kernels.h"
#include "stream_probe.h"
#include "wkv_tiles.cuh"

namespace engram {

namespace {

constexpr int kProbeStages = 6;
constexpr uint32_t kProbeChunk = 32 * 1024;
constexpr int kPlainThreads = 512;

struct ProbeShared {
  uint64_t full[kProbeStages];
  int abort;
};

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_load_hint(void* dst, const void* src, uint32_t bytes,
                                               uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// share of CTA b of n over `units` 16-byte units: [lo, hi)
__device__ __forceinline__ void cta_share(int64_t units, int64_t& lo, int64_t& hi) {
  lo = units * blockIdx.x / gridDim.x;
  hi = units * (blockIdx.x + 1) / gridDim.x;
}

__global__ void __launch_bounds__(32, 1) probe_bulk_kernel(const uint8_t* src, int64_t units,
                                                           int32_t evict_first, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = align_1024(smem_raw);
  ProbeShared* sh = reinterpret_cast<ProbeShared*>(ring + kProbeStages * kProbeChunk);
  if (threadIdx.x != 0) return;
  for (int i = 0; i < kProbeStages; ++i) mbar_init(&sh->full[i], 1);
  sh->abort = 0;
  fence_mbar_init();
  int64_t lo, hi;
  cta_share(units, lo, hi);
  const uint8_t* p = src + lo * 16;
  const int64_t bytes = (hi - lo) * 16;
  const int64_t chunks = (bytes + kProbeChunk - 1) / kProbeChunk;
  volatile int* abort = &sh->abort;
  int64_t issued = 0;
  for (int64_t c = 0; c < chunks; ++c) {
    const int stage = static_cast<int>(c % kProbeStages);
    if (c >= kProbeStages) {   // the stage's previous chunk has landed before it is refilled
      const uint32_t parity = static_cast<uint32_t>((c / kProbeStages - 1) & 1);
      if (!mbar_wait(&sh->full[stage], parity, abort, err)) break;
    }
    const int64_t left = bytes - c * kProbeChunk;
    const uint32_t n = static_cast<uint32_t>(left < kProbeChunk ? left : kProbeChunk);
    mbar_arrive_expect_tx(&sh->full[stage], n);
    if (evict_first)
      bulk_load_hint(ring + stage * kProbeChunk, p + c * kProbeChunk, n, &sh->full[stage],
                     l2_evict_first_policy());
    else
      bulk_load(ring + stage * kProbeChunk, p + c * kProbeChunk, n, &sh->full[stage]);
    issued = c + 1;
  }
  // every copy issued has landed before the CTA exits (each stage's last fill; bounded)
  for (int64_t c = issued - kProbeStages < 0 ? 0 : issued - kProbeStages; c < issued; ++c)
    mbar_wait_drain(&sh->full[c % kProbeStages], static_cast<uint32_t>((c / kProbeStages) & 1));
}

__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// where the plain loads' fold is written, for one value in 2^32 only; never read
__device__ uint32_t g_probe_sink;

__global__ void __launch_bounds__(kPlainThreads) probe_plain_kernel(const uint8_t* src,
                                                                    int64_t units) {
  int64_t lo, hi;
  cta_share(units, lo, hi);
  const uint4* p = reinterpret_cast<const uint4*>(src);
  uint32_t x = 0;
  int64_t i = lo + threadIdx.x;
  for (; i + 3 * kPlainThreads < hi; i += 4 * kPlainThreads) {
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = ldg_stream(p + i + j * kPlainThreads);
#pragma unroll
    for (int j = 0; j < 4; ++j) x ^= v[j].x ^ v[j].y ^ v[j].z ^ v[j].w;
  }
  for (; i < hi; i += kPlainThreads) {
    const uint4 v = ldg_stream(p + i);
    x ^= v.x ^ v.y ^ v.z ^ v.w;
  }
  x = __reduce_xor_sync(0xFFFFFFFFu, x);
  if ((threadIdx.x & 31) == 0 && x == 0x9E3779B9u) atomicXor(&g_probe_sink, x);   // keeps the loads live
}

}  // namespace

size_t probe_bulk_smem_bytes() {
  return size_t(kProbeStages) * kProbeChunk + sizeof(ProbeShared) + 1024;
}

cudaError_t launch_stream_probe(const void* src, int64_t bytes, int32_t method, uint32_t* err,
                                cudaStream_t st) {
  const int64_t units = bytes / 16;
  const unsigned grid = static_cast<unsigned>(device_sm_count());
  if (method == kProbeBulk || method == kProbeBulkEvictFirst) {
    const size_t smem = probe_bulk_smem_bytes();
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(probe_bulk_kernel), smem);
    if (e != cudaSuccess) return e;
    probe_bulk_kernel<<<grid, 32, smem, st>>>(static_cast<const uint8_t*>(src), units,
                                              method == kProbeBulkEvictFirst, err);
  } else {
    probe_plain_kernel<<<grid, kPlainThreads, 0, st>>>(static_cast<const uint8_t*>(src), units);
  }
  return cudaGetLastError();
}

}  // namespace engram
