// fd_copy.h - launcher of the one-kernel copy (fd_copy.cu) used by the C-ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace fd {

// One-kernel copy of `bytes` (multiple of 16) between device-accessible buffers; falls
// back to cudaMemcpyAsync when either side is not accessible to a kernel.
cudaError_t launch_copy(void *dst, const void *src, size_t bytes, cudaStream_t stream);

}  // namespace fd
