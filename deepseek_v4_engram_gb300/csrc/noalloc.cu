// engram_forward_noalloc: engram_forward for callers that cannot allocate device memory.
//
// Some callers cannot hand this library a workspace: a runtime that owns all device memory and
// gives a plugin only its input and output buffers, or a serving loop that must never call
// cudaMalloc (which can synchronise the whole device) once it is running. For them this entry
// point runs the same kernels as engram_forward, with the scratch (hash ids and gathered rows)
// in a fixed array in device memory that belongs to the library itself.
#include <cstdio>
#include <mutex>

#include "engram.h"
#include "kernels.h"

namespace engram {
namespace {

// The library's own scratch: ENGRAM_NOALLOC_SCRATCH_BYTES bytes, in every GPU that loads the
// library, until the process exits. Every call shares it.
static __device__ __align__(256) uint8_t g_forward_scratch[ENGRAM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's copy of the scratch array. In host code the array's name
// stands for a host-side shadow, not a device address, so the address comes from the runtime,
// once per device, with that device current.
void* scratch_address(cudaError_t* err) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = e != cudaSuccess ? e : cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_forward_scratch);
    if (e != cudaSuccess || p == nullptr) {
      *err = e != cudaSuccess ? e : cudaErrorInvalidSymbol;
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  *err = cudaSuccess;
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace engram

using namespace engram;

extern "C" ENGRAM_API int engram_forward_noalloc(
    const engram_desc_t* desc, const engram_tables_t* tables, const engram_weights_t* weights,
    const uint16_t* x, const int32_t* tokens, int32_t B, int32_t T, int32_t* cache,
    int32_t* cache_len, int32_t capacity, const uint8_t* token_mask, uint16_t* out,
    int32_t* hash_ids_out, float* gate_out, uint16_t* kv_out, void* stream) {
  if (B < 0 || T < 0) return set_last_error(ENGRAM_EINVAL, "B and T must be >= 0");
  const int64_t M = int64_t(B) * T;
  // engram_forward runs the fastest path whose scratch fits; the smallest one must fit here
  const size_t need = forward_min_workspace_bytes(desc, M);
  if (need == 0 && M > 0) return set_last_error(ENGRAM_EINVAL, "invalid engram_desc_t");
  if (need > size_t(ENGRAM_NOALLOC_SCRATCH_BYTES)) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "engram_forward_noalloc: %lld tokens need %zu bytes of scratch, more than the %d "
             "bytes it owns; split the call or use engram_forward with a workspace",
             static_cast<long long>(M), need, ENGRAM_NOALLOC_SCRATCH_BYTES);
    return set_last_error(ENGRAM_EINVAL, msg);
  }
  cudaError_t e;
  void* scratch = scratch_address(&e);
  if (scratch == nullptr) {
    char msg[256];
    snprintf(msg, sizeof(msg), "engram_forward_noalloc: scratch address: %s",
             cudaGetErrorString(e));
    return set_last_error(ENGRAM_ECUDA, msg);
  }
  return engram_forward(desc, tables, weights, x, tokens, B, T, cache, cache_len, capacity,
                        token_mask, out, hash_ids_out, gate_out, kv_out, scratch,
                        size_t(ENGRAM_NOALLOC_SCRATCH_BYTES), stream);
}
