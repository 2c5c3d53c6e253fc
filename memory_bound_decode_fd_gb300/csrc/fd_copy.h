// fd_copy.h - launcher of the one-kernel copy (fd_copy.cu) used by the C-ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace fd {

// One-kernel copy of `bytes` (multiple of 16) between device-accessible buffers; falls
// back to cudaMemcpyAsync when either side is not accessible to a kernel.
cudaError_t launch_copy(void *dst, const void *src, size_t bytes, cudaStream_t stream);

// The same for `rows` rows of `row_bytes` (multiple of 16) at pitches dst_pitch and
// src_pitch (multiples of 16); falls back to cudaMemcpy2DAsync.
cudaError_t launch_copy_rows(void *dst, size_t dst_pitch, const void *src, size_t src_pitch,
                             size_t row_bytes, size_t rows, cudaStream_t stream);

}  // namespace fd
