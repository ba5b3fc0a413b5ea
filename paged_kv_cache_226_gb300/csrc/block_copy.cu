// Whole-block copies between block pools: copy-on-write of a shared block
// and swapping blocks between the device pool and a pinned host pool.
//
// Copy-on-write: requests that share physical blocks (parallel sampling,
// beam search, a common prompt) keep sharing them until one must write into
// a shared block; that request then gets a private copy (tcdigital article,
// section on memory sharing for parallel sampling; youngju.dev post,
// Copy-on-Write prefix sharing).  Swapping: a preempted request's blocks can
// move to CPU memory and back (tcdigital article, --swap-space; ta-paperlens
// scheduler skeleton, preemption by moving to the CPU or recomputing).
#include "pa_device.cuh"

namespace pa {

// One CTA moves one 16 KiB chunk of one block of K or V with 16-byte
// vectors.  grid = (chunks per block, 2 (K, V), pairs).
constexpr int kCopyChunkBytes = 16384;
constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads)
    copy_blocks_kernel(const uint4* __restrict__ k_src, const uint4* __restrict__ v_src,
                       int64_t src_blocks, uint4* __restrict__ k_dst, uint4* __restrict__ v_dst,
                       int64_t dst_blocks, const int64_t* __restrict__ mapping,
                       int64_t vec_per_block, int* err) {
    grid_dependency_wait();
    allow_dependent_launch();
    const int64_t pair = blockIdx.z;
    const int64_t src = mapping[2 * pair];
    const int64_t dst = mapping[2 * pair + 1];
    if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
            flag_error(err, PA_DEVERR_BAD_SLOT);
        return;
    }
    const uint4* s = (blockIdx.y == 0 ? k_src : v_src) + src * vec_per_block;
    uint4* d = (blockIdx.y == 0 ? k_dst : v_dst) + dst * vec_per_block;
    const int64_t begin = (int64_t)blockIdx.x * (kCopyChunkBytes / 16);
    const int64_t end = min(begin + kCopyChunkBytes / 16, vec_per_block);
    int64_t i = begin + threadIdx.x;
    // four vectors in flight per thread
    for (; i + 3 * kCopyThreads < end; i += 4 * kCopyThreads) {
        const uint4 a = s[i];
        const uint4 b = s[i + kCopyThreads];
        const uint4 c = s[i + 2 * kCopyThreads];
        const uint4 e = s[i + 3 * kCopyThreads];
        d[i] = a;
        d[i + kCopyThreads] = b;
        d[i + 2 * kCopyThreads] = c;
        d[i + 3 * kCopyThreads] = e;
    }
    for (; i < end; i += kCopyThreads) d[i] = s[i];
}

cudaError_t launch_copy_blocks(const void* k_src, const void* v_src, int64_t src_blocks,
                               void* k_dst, void* v_dst, int64_t dst_blocks,
                               const int64_t* mapping, int64_t num_pairs, int64_t block_bytes,
                               int* err, cudaStream_t stream) {
    const unsigned chunks = (unsigned)((block_bytes + kCopyChunkBytes - 1) / kCopyChunkBytes);
    return launch_with_pdl(copy_blocks_kernel, dim3(chunks, 2, (unsigned)num_pairs),
                           dim3(kCopyThreads), 0, stream, static_cast<const uint4*>(k_src),
                           static_cast<const uint4*>(v_src), src_blocks,
                           static_cast<uint4*>(k_dst), static_cast<uint4*>(v_dst), dst_blocks,
                           mapping, block_bytes / 16, err);
}

}  // namespace pa
