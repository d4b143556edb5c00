// Staging copy between device and pinned host memory (append.cu), behind kvc_copy_async.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>

namespace kvc {
// bytes > 0 and a multiple of 16; both addresses 16-byte aligned device addresses (pinned host memory through
// its mapping).  ahead: copy alongside the kernel before on the stream (the KVC_COPY_AHEAD ordering).
cudaError_t launch_stage_copy(void* dst, const void* src, size_t bytes, bool ahead, cudaStream_t stream);
}  // namespace kvc
