// Byte copies by SMs, for a layer-step's small host <-> device transfers: the
// inputs come from pinned host memory and the output goes back to it through
// unified addressing (device loads and stores reach pinned host memory
// directly), in one short launch that chains to the step kernels with
// programmatic dependent launch instead of a copy-engine transfer.
#include "pa_internal.h"
#include "pa_device.cuh"

namespace pa {

__global__ void __launch_bounds__(256) copy16_kernel(uint4* __restrict__ dst,
                                                     const uint4* __restrict__ src, size_t n16) {
    grid_dependency_wait();          // src may be written by the previous kernel
    allow_dependent_launch();
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    // four 16-byte loads in flight per thread
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride],
                    d = src[i + 3 * stride];
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = d;
    }
    for (; i < n16; i += stride) dst[i] = src[i];
}

cudaError_t launch_copy16(void* dst, const void* src, size_t n16, cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const size_t want = (n16 + 4 * 256 - 1) / (4 * 256);
    const unsigned blocks = (unsigned)(want < 1 ? 1 : (want > (size_t)sms * 4 ? (size_t)sms * 4 : want));
    return launch_with_pdl(copy16_kernel, dim3(blocks), dim3(256), 0, stream,
                           static_cast<uint4*>(dst), static_cast<const uint4*>(src), n16);
}

}  // namespace pa
