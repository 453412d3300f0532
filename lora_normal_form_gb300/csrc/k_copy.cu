// Gather and scatter of a batched call's host buffers through the device's
// mapping of pinned host memory.
//
// scute_linear_batch_host moves every call's input rows to the device and
// every call's output rows back.  When each of those host buffers is pinned
// and mapped, one launch copies all of them (the kernel reads or writes the
// host memory through its device address) instead of one copy per buffer:
// each copy pays its own setup, while here the buffers share one launch.
#include "internal.h"

namespace scute {

namespace {

__global__ void __launch_bounds__(256) copy_segments_kernel(const __grid_constant__ CopySegs s) {
    const int i = blockIdx.y;
    if (i >= s.n) return;
    const uint8_t *src = reinterpret_cast<const uint8_t *>(s.src[i]);
    uint8_t *dst = reinterpret_cast<uint8_t *>(s.dst[i]);
    const size_t bytes = s.bytes[i];
    const size_t step = (size_t)gridDim.x * blockDim.x;
    const size_t t0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    size_t done = 0;
    if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u) == 0) {
        const size_t n16 = bytes / 16;
        const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
        for (size_t k = t0; k < n16; k += step) d4[k] = s4[k];
        done = n16 * 16;
    }
    for (size_t k = done + t0; k < bytes; k += step) dst[k] = src[k];
}

}  // namespace

cudaError_t launch_copy_segments(const CopySegs &s, cudaStream_t st) {
    if (s.n <= 0) return cudaSuccess;
    size_t most = 0;
    for (int i = 0; i < s.n; ++i) most = s.bytes[i] > most ? s.bytes[i] : most;
    // about 16 KB per CTA of the largest buffer, at least one CTA
    size_t bx = (most + 16383) / 16384;
    if (bx < 1) bx = 1;
    if (bx > 256) bx = 256;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)bx, (unsigned)s.n, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, copy_segments_kernel, s);
}

}  // namespace scute
