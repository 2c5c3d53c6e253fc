// fd_copy.cu - one-kernel copy between device-accessible buffers, for the per-token I/O of
// a decode step. On GB300 (Grace + Blackwell) pinned host memory is read and written by
// the GPU over NVLink-C2C. Alone, a copy-engine transfer of a step's 1.85 MB of inputs
// (32 layers of gate/up at MLP width 14336) takes about as long as this kernel (10.7 vs
// 13.1 us), but inside the captured step the kernels overlap their neighbours under
// programmatic dependent launch: the step's end-to-end time measured 321 us with them
// against 335 us with copy-engine transfers (memcpy nodes) for the same two copies.
#include "fd_copy.h"
#include "fd_internal.h"

namespace fd {
namespace {

// 16-byte vectors, grid-stride; waits for the previous kernel in the stream first (the
// source may be its output) when launched with programmatic dependent launch.
__global__ void __launch_bounds__(256) copy_kernel(const uint4 *__restrict__ src,
                                                   uint4 *__restrict__ dst, size_t n16) {
    grid_dep_wait();
    grid_dep_launch();
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = d;
    }
    for (; i < n16; i += stride) dst[i] = src[i];
}

// Rows of n16 16-byte vectors at pitches dp16 and sp16 (in vectors), grid-stride over all
// vectors of all rows.
__global__ void __launch_bounds__(256) copy_rows_kernel(const uint4 *__restrict__ src,
                                                        uint4 *__restrict__ dst, size_t n16,
                                                        size_t rows, size_t sp16, size_t dp16) {
    grid_dep_wait();
    grid_dep_launch();
    const size_t total = n16 * rows;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        const size_t r = i / n16, c = i - r * n16;
        dst[r * dp16 + c] = src[r * sp16 + c];
    }
}

// The device address of `p` if the GPU can access it (device, managed, or mapped pinned
// host memory), else nullptr.
const void *device_address(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error of an unknown pointer
        return nullptr;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return p;
    if (a.type == cudaMemoryTypeHost) return a.devicePointer;
    return nullptr;
}

long long copy_blocks(size_t n16, int sm_count) {
    long long blocks = (long long)((n16 + 255) / 256);
    const long long cap = (long long)sm_count * 4;
    if (blocks > cap) blocks = cap;
    return blocks < 1 ? 1 : blocks;
}

}  // namespace

cudaError_t launch_copy_rows(void *dst, size_t dst_pitch, const void *src, size_t src_pitch,
                             size_t row_bytes, size_t rows, cudaStream_t stream) {
    const void *s = device_address(src);
    void *d = const_cast<void *>(device_address(dst));
    if (!s || !d)
        return cudaMemcpy2DAsync(dst, dst_pitch, src, src_pitch, row_bytes, rows,
                                 cudaMemcpyDefault, stream);
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    const size_t n16 = row_bytes / 16;
    err = launch_kernel(copy_rows_kernel, dim3((unsigned)copy_blocks(n16 * rows, di.sm_count)),
                        dim3(256), 0, stream, 1, static_cast<const uint4 *>(s),
                        static_cast<uint4 *>(d), n16, rows, src_pitch / 16, dst_pitch / 16);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

cudaError_t launch_copy(void *dst, const void *src, size_t bytes, cudaStream_t stream) {
    const void *s = device_address(src);
    void *d = const_cast<void *>(device_address(dst));
    if (!s || !d) {
        // not accessible to a kernel (e.g. pageable host memory): the copy engine
        return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, stream);
    }
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    const size_t n16 = bytes / 16;
    long long blocks = (long long)((n16 + 255) / 256);
    const long long cap = (long long)di.sm_count * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    err = launch_kernel(copy_kernel, dim3((unsigned)blocks), dim3(256), 0, stream, 1,
                        static_cast<const uint4 *>(s), static_cast<uint4 *>(d), n16);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace fd
