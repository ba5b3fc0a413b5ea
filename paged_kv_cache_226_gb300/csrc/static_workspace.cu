// pa_decode_static_workspace: the split decode + merge with its partition
// workspace in a fixed device buffer owned by the library, for callers that
// cannot allocate device memory themselves.
//
// Who needs it: code that runs where a cudaMalloc is not allowed or not
// wanted -- a plug-in inside an inference server whose device memory is
// owned by the host framework's pool (a private cudaMalloc would bypass the
// pool's accounting and can fail once the pool has taken the free memory),
// or a latency-critical loop that cannot afford the implicit device-wide
// synchronisation of cudaMalloc / cudaFree.  Such callers pass only their
// inputs and their output; the partition buffers come from here.
#include <cuda_runtime.h>

#include <mutex>

#include "pa_internal.h"

namespace {

// The buffer: PA_STATIC_WORKSPACE_BYTES of device memory on every GPU that
// loads the library, held until the process exits.
__device__ __align__(256) unsigned char g_static_workspace[PA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
// The buffer's device address per device, with the context it was looked up
// in: a __device__ array's address belongs to a CUDA context, so a call made
// under another context (a driver-API context, or the primary context made
// anew after cudaDeviceReset) looks it up again instead of reusing an
// address that context never mapped.
struct Slot {
    void* ctx;
    void* ptr;
};
Slot g_workspace_slot[kMaxDevices];
std::mutex g_workspace_mutex;

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Device address of the buffer on the current device and context.  The
// first call there looks it up (cudaGetSymbolAddress, which also loads the
// module holding the buffer); later calls under the same context reuse it.
cudaError_t workspace_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void* ctx = nullptr;
    if ((e = pa::current_context(&ctx)) != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_workspace_mutex);
    Slot& slot = g_workspace_slot[dev];
    if (slot.ptr == nullptr || ctx == nullptr || slot.ctx != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_workspace);
        if (e != cudaSuccess) return e;
        if ((e = pa::current_context(&ctx)) != cudaSuccess) return e;   // made current above
        slot.ctx = ctx;
        slot.ptr = p;
    }
    *out = slot.ptr;
    return cudaSuccess;
}

}  // namespace

extern "C" int pa_decode_static_workspace(const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* block_tables,
                                          const int32_t* context_lens, float scale,
                                          int32_t partition_size, int32_t max_num_partitions,
                                          void* out, const pa_shape* shp, void* stream) {
    // the argument checks of pa_decode_split + pa_reduce come first, so a
    // malformed request gets the status those entry points give it
    const int st0 = pa::check_split_request(q, k_cache, v_cache, block_tables, context_lens,
                                            partition_size, max_num_partitions, out, shp);
    if (st0 != PA_OK) return st0;
    if (shp->num_seqs == 0) return PA_OK;
    // tmp_out [B][Hq][S][D], then max_logits and exp_sums [B][Hq][S], fp32,
    // each part starting on a 256-byte boundary.
    const size_t rows = (size_t)shp->num_seqs * shp->num_q_heads * (size_t)max_num_partitions;
    const size_t tmp_bytes = round256(rows * shp->head_dim * sizeof(float));
    const size_t vec_bytes = round256(rows * sizeof(float));
    if (tmp_bytes + 2 * vec_bytes > (size_t)PA_STATIC_WORKSPACE_BYTES) return PA_ERR_WORKSPACE;
    void* base = nullptr;
    cudaError_t e = workspace_address(&base);
    if (e != cudaSuccess) {
        pa::record_cuda_error(static_cast<int>(e));
        return PA_ERR_CUDA;
    }
    float* tmp_out = static_cast<float*>(base);
    float* max_logits = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + tmp_bytes);
    float* exp_sums = reinterpret_cast<float*>(static_cast<unsigned char*>(base) + tmp_bytes +
                                               vec_bytes);
    // Nothing in the buffer needs clearing: the merge reads exactly the
    // partitions that the split kernel of this same call writes.
    int st = pa_decode_split(q, k_cache, v_cache, block_tables, context_lens, scale,
                             partition_size, max_num_partitions, tmp_out, max_logits, exp_sums,
                             shp, stream);
    if (st != PA_OK) return st;
    return pa_reduce(tmp_out, max_logits, exp_sums, context_lens, partition_size,
                     max_num_partitions, out, shp, stream);
}
