// A one-pass read of a device buffer over every SM (a measured floor for weight-streaming
// kernels); see stream_probe.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace engram {

enum : int32_t { kProbeBulk = 0, kProbePlain = 1, kProbeBulkEvictFirst = 2 };

cudaError_t launch_stream_probe(const void* src, int64_t bytes, int32_t method, uint32_t* err,
                                cudaStream_t st);

}  // namespace engram
