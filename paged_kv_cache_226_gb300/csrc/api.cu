// C-ABI entry points of libpa.so: host-side validation, TMA descriptor
// encoding and kernel dispatch.  Declarations and contracts: include/pa.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pa_internal.h"
#include "prefill_internal.h"

namespace {

// Device error word (PA_DEVERR_* bits), one per device the library runs on.
__device__ int g_device_errors;

constexpr int kMaxDevices = 64;
// Its address, looked up per device and remembered with the context it was
// looked up in: a __device__ variable's address belongs to a context, so a
// different current context (a driver-API context, or the primary context
// re-created after cudaDeviceReset) triggers a fresh lookup.
struct SymbolSlot {
    void* ctx;
    int* ptr;
};
SymbolSlot g_err_slot[kMaxDevices];
std::mutex g_err_mutex;
thread_local int t_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return PA_ERR_CUDA;
}

// cuCtxGetCurrent through the runtime's driver entry point (no link
// dependency on libcuda).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
CtxGetCurrentFn g_ctx_get = nullptr;
std::once_flag g_ctx_once;
cudaError_t g_ctx_status = cudaSuccess;

// Device address of the error word on the current device.
cudaError_t error_word(int** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void* ctx = nullptr;
    if ((e = pa::current_context(&ctx)) != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_err_mutex);
    SymbolSlot& slot = g_err_slot[dev];
    if (slot.ptr == nullptr || ctx == nullptr || slot.ctx != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_errors);   // makes a context current if none is
        if (e != cudaSuccess) return e;
        if ((e = pa::current_context(&ctx)) != cudaSuccess) return e;
        slot.ctx = ctx;
        slot.ptr = static_cast<int*>(p);
    }
    *out = slot.ptr;
    return cudaSuccess;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_status = cudaSuccess;

cudaError_t get_encoder(EncodeTiledFn* fn) {
    std::call_once(g_encode_once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                                         cudaEnableDefault, &q);
        if (e == cudaSuccess && (q != cudaDriverEntryPointSuccess || p == nullptr))
            e = cudaErrorSymbolNotFound;
        g_encode_status = e;
        g_encode = reinterpret_cast<EncodeTiledFn>(p);
    });
    *fn = g_encode;
    return g_encode_status;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Common shape checks.  Returns PA_OK or an error status.
int check_shape(const pa_shape* s, bool need_q_heads) {
    if (s == nullptr) return PA_ERR_INVALID_ARG;
    if (s->reserved != 0) return PA_ERR_INVALID_ARG;
    if (s->dtype != PA_FP16 && s->dtype != PA_BF16) return PA_ERR_INVALID_ARG;
    if (s->num_kv_heads <= 0 || s->head_dim <= 0 || s->block_size <= 0 || s->num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (s->head_dim != 64 && s->head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (s->block_size != 16 && s->block_size != 32) return PA_ERR_UNSUPPORTED;
    if (s->num_blocks > 0xffffffffll) return PA_ERR_UNSUPPORTED;
    if (need_q_heads) {
        if (s->num_seqs < 0 || s->num_seqs > 65535) return PA_ERR_INVALID_ARG;
        if (s->num_q_heads <= 0 || s->num_q_heads % s->num_kv_heads != 0)
            return PA_ERR_INVALID_ARG;
        if (s->num_q_heads / s->num_kv_heads > pa::kMaxGroup) return PA_ERR_UNSUPPORTED;
        if (s->num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
        if (s->max_blocks_per_seq <= 0) return PA_ERR_INVALID_ARG;
        if ((int64_t)s->max_blocks_per_seq * s->block_size > (1ll << 30)) return PA_ERR_UNSUPPORTED;
    }
    return PA_OK;
}

// 4-D view [num_blocks][block_size][Hkv][D] of a cache; box = one 128-byte
// row slice (64 dims of a 16-bit cache, 128 dims of an FP8 one) x one head x
// 16 tokens x one block, 128 B swizzle (conflict-free ldmatrix rows).
int encode_cache_map(CUtensorMap* map, const void* base, const pa_shape* s, bool fp8) {
    EncodeTiledFn enc = nullptr;
    cudaError_t e = get_encoder(&enc);
    if (e != cudaSuccess) return cuda_fail(e);
    const cuuint64_t elem = fp8 ? 1 : 2;
    cuuint64_t dims[4] = {(cuuint64_t)s->head_dim, (cuuint64_t)s->num_kv_heads,
                          (cuuint64_t)s->block_size, (cuuint64_t)s->num_blocks};
    cuuint64_t strides[3] = {s->head_dim * elem, (cuuint64_t)s->num_kv_heads * s->head_dim * elem,
                             (cuuint64_t)s->block_size * s->num_kv_heads * s->head_dim * elem};
    cuuint32_t box[4] = {(cuuint32_t)(128 / elem), 1, (cuuint32_t)pa::kTileTokens, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : (s->dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
    CUresult r = enc(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return PA_ERR_INVALID_ARG;
    return PA_OK;
}

// How the cache stores K and V: the 16-bit type of shp->dtype, or E4M3 bytes
// with per-tensor scales.
struct CacheKind {
    bool fp8;
    float k_scale;
    float v_scale;
};
constexpr CacheKind kCache16 = {false, 1.f, 1.f};

int check_decode_args(const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens,
                      const pa_shape* shp) {
    int st = check_shape(shp, true);
    if (st != PA_OK) return st;
    if (shp->num_seqs == 0) return PA_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(block_tables) ||
        !aligned16(context_lens))
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

#ifdef PA_TEST_HOOKS
// Test builds only: the wait fault of pa_test_set_wait_fault (none by default).
int g_test_cta = -1;
int g_test_tile = 0;
unsigned long long g_test_wait_limit_ns = pa::kWaitLimitNs;
#endif

pa::DecodeParams make_params(const void* q, const int32_t* block_tables,
                             const int32_t* context_lens, float scale, const pa_shape* shp,
                             int* err, const CacheKind& ck) {
    pa::DecodeParams p{};
    p.q = q;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.err = err;
    p.scale_log2 = scale * ck.k_scale * pa::kLog2e;
    p.k_scale = ck.k_scale;
    p.v_scale = ck.v_scale;
    p.num_q_heads = shp->num_q_heads;
    p.group = shp->num_q_heads / shp->num_kv_heads;
    p.max_blocks_per_seq = shp->max_blocks_per_seq;
    p.block_size = shp->block_size;
    p.num_blocks = shp->num_blocks;
    p.num_kv_heads = shp->num_kv_heads;
#ifdef PA_TEST_HOOKS
    p.test_cta = g_test_cta;
    p.test_tile = g_test_tile;
    p.test_wait_limit_ns = g_test_wait_limit_ns;
#endif
    return p;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

void pa::record_cuda_error(int cuda_error) { t_last_cuda_error = cuda_error; }

cudaError_t pa::current_context(void** ctx) {
    std::call_once(g_ctx_once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000,
                                                         cudaEnableDefault, &q);
        if (e == cudaSuccess && (q != cudaDriverEntryPointSuccess || p == nullptr))
            e = cudaErrorSymbolNotFound;
        g_ctx_status = e;
        g_ctx_get = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    if (g_ctx_status != cudaSuccess) return g_ctx_status;
    CUcontext c = nullptr;
    if (g_ctx_get(&c) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;   // "invalid device context"
    *ctx = static_cast<void*>(c);
    return cudaSuccess;
}

int pa::check_split_request(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens,
                            int32_t partition_size, int32_t max_num_partitions, const void* out,
                            const pa_shape* shp) {
    // the checks of pa_decode_split (16-bit cache), then those of pa_reduce
    // on its output, in the order those entry points run them
    int st = check_decode_args(q, k_cache, v_cache, block_tables, context_lens, shp);
    if (st != PA_OK) return st;
    if (partition_size <= 0 || partition_size % shp->block_size != 0) return PA_ERR_INVALID_ARG;
    if (max_num_partitions <= 0) return PA_ERR_WORKSPACE;
    if (max_num_partitions > 65535) return PA_ERR_UNSUPPORTED;
    if (shp->num_seqs == 0) return PA_OK;
    if (!out || !aligned16(out)) return PA_ERR_INVALID_ARG;
    return PA_OK;
}

extern "C" {

const char* pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape";
        case PA_ERR_WORKSPACE: return "split workspace too small";
        case PA_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

int pa_last_cuda_error(void) { return t_last_cuda_error; }

#ifdef PA_TEST_HOOKS
int pa_test_set_wait_fault(int32_t cta, int32_t tile, unsigned long long wait_limit_ns) {
    if (wait_limit_ns == 0) return PA_ERR_INVALID_ARG;
    g_test_cta = cta;
    g_test_tile = tile;
    g_test_wait_limit_ns = wait_limit_ns;
    return PA_OK;
}
#endif

int pa_read_device_errors(int32_t* flags, void* stream) {
    if (flags == nullptr) return PA_ERR_INVALID_ARG;
    int* err = nullptr;
    cudaError_t e = error_word(&err);
    if (e != cudaSuccess) return cuda_fail(e);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int host = 0;
    e = cudaMemcpyAsync(&host, err, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(err, 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    *flags = host;
    return PA_OK;
}

int pa_reshape_and_cache(const void* k, const void* v, const int64_t* slot_mapping,
                         void* k_cache, void* v_cache, int64_t num_tokens,
                         const pa_shape* shp, void* stream) {
    int st = check_shape(shp, false);
    if (st != PA_OK) return st;
    if (num_tokens < 0 || num_tokens > 0x7fffffffll) return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PA_ERR_INVALID_ARG;
    int* err = nullptr;
    cudaError_t e = error_word(&err);
    if (e != cudaSuccess) return cuda_fail(e);
    const int row_bytes = shp->num_kv_heads * shp->head_dim * 2;
    e = pa::launch_reshape_and_cache(k, v, slot_mapping, k_cache, v_cache, num_tokens,
                                     shp->num_blocks * shp->block_size, row_bytes, err,
                                     static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

}  // extern "C"

namespace {

int check_kind(const pa_shape* shp, const CacheKind& ck) {
    if (!ck.fp8) return PA_OK;
    if (shp->head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (!(ck.k_scale > 0.f) || !(ck.v_scale > 0.f) || ck.k_scale == INFINITY ||
        ck.v_scale == INFINITY)
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

cudaError_t launch(int mode, const pa_shape* shp, const CacheKind& ck, const CUtensorMap& tmk,
                   const CUtensorMap& tmv, const pa::DecodeParams& p, dim3 grid, void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (ck.fp8) return pa::launch_decode_fp8(shp->dtype, mode, tmk, tmv, p, grid, s);
    return pa::launch_decode(shp->dtype, shp->head_dim, mode, tmk, tmv, p, grid, s);
}

int decode_single(const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens, float scale,
                  void* out, const pa_shape* shp, void* stream, const CacheKind& ck) {
    int st = check_decode_args(q, k_cache, v_cache, block_tables, context_lens, shp);
    if (st != PA_OK) return st;
    if ((st = check_kind(shp, ck)) != PA_OK) return st;
    if (shp->num_seqs == 0) return PA_OK;
    if (!out || !aligned16(out)) return PA_ERR_INVALID_ARG;
    CUtensorMap tmk, tmv;
    if ((st = encode_cache_map(&tmk, k_cache, shp, ck.fp8)) != PA_OK) return st;
    if ((st = encode_cache_map(&tmv, v_cache, shp, ck.fp8)) != PA_OK) return st;
    int* err = nullptr;
    cudaError_t e = error_word(&err);
    if (e != cudaSuccess) return cuda_fail(e);
    pa::DecodeParams p = make_params(q, block_tables, context_lens, scale, shp, err, ck);
    p.out = out;
    dim3 grid(shp->num_seqs, shp->num_kv_heads, 1);
    e = launch(pa::kModeSingle, shp, ck, tmk, tmv, p, grid, stream);
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int decode_split(const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* block_tables, const int32_t* context_lens, float scale,
                 int32_t partition_size, int32_t max_num_partitions, float* tmp_out,
                 float* max_logits, float* exp_sums, const pa_shape* shp, void* stream,
                 const CacheKind& ck) {
    int st = check_decode_args(q, k_cache, v_cache, block_tables, context_lens, shp);
    if (st != PA_OK) return st;
    if ((st = check_kind(shp, ck)) != PA_OK) return st;
    if (partition_size <= 0 || partition_size % shp->block_size != 0) return PA_ERR_INVALID_ARG;
    if (max_num_partitions <= 0) return PA_ERR_WORKSPACE;
    if (max_num_partitions > 65535) return PA_ERR_UNSUPPORTED;
    if (shp->num_seqs == 0) return PA_OK;
    if (!tmp_out || !max_logits || !exp_sums) return PA_ERR_WORKSPACE;
    if (!aligned16(tmp_out) || !aligned16(max_logits) || !aligned16(exp_sums))
        return PA_ERR_INVALID_ARG;
    CUtensorMap tmk, tmv;
    if ((st = encode_cache_map(&tmk, k_cache, shp, ck.fp8)) != PA_OK) return st;
    if ((st = encode_cache_map(&tmv, v_cache, shp, ck.fp8)) != PA_OK) return st;
    int* err = nullptr;
    cudaError_t e = error_word(&err);
    if (e != cudaSuccess) return cuda_fail(e);
    pa::DecodeParams p = make_params(q, block_tables, context_lens, scale, shp, err, ck);
    p.tmp_out = tmp_out;
    p.max_logits = max_logits;
    p.exp_sums = exp_sums;
    p.partition_tokens = partition_size;
    p.max_parts = max_num_partitions;
    dim3 grid(shp->num_seqs, shp->num_kv_heads, max_num_partitions);
    e = launch(pa::kModeSplit, shp, ck, tmk, tmv, p, grid, stream);
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int decode_step(const void* q, const void* k, const void* v, const int64_t* slot_mapping,
                void* k_cache, void* v_cache, const int32_t* block_tables,
                const int32_t* context_lens, float scale, int32_t partition_size,
                int32_t max_num_partitions, float* tmp_out, float* max_logits, float* exp_sums,
                int32_t* counters, void* out, const pa_shape* shp, void* stream,
                const CacheKind& ck) {
    int st = check_decode_args(q, k_cache, v_cache, block_tables, context_lens, shp);
    if (st != PA_OK) return st;
    if ((st = check_kind(shp, ck)) != PA_OK) return st;
    if (partition_size <= 0 || partition_size % shp->block_size != 0) return PA_ERR_INVALID_ARG;
    if (max_num_partitions <= 0) return PA_ERR_WORKSPACE;
    if (shp->num_seqs == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !out || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PA_ERR_INVALID_ARG;
    if (!tmp_out || !max_logits || !exp_sums || !counters) return PA_ERR_WORKSPACE;
    if (!aligned16(tmp_out) || !aligned16(max_logits) || !aligned16(exp_sums) ||
        (reinterpret_cast<uintptr_t>(counters) & 3u))
        return PA_ERR_INVALID_ARG;
    CUtensorMap tmk, tmv;
    if ((st = encode_cache_map(&tmk, k_cache, shp, ck.fp8)) != PA_OK) return st;
    if ((st = encode_cache_map(&tmv, v_cache, shp, ck.fp8)) != PA_OK) return st;
    int* err = nullptr;
    cudaError_t e = error_word(&err);
    if (e != cudaSuccess) return cuda_fail(e);
    pa::DecodeParams p = make_params(q, block_tables, context_lens, scale, shp, err, ck);
    p.out = out;
    p.tmp_out = tmp_out;
    p.max_logits = max_logits;
    p.exp_sums = exp_sums;
    p.partition_tokens = partition_size;
    p.max_parts = max_num_partitions;
    p.k_new = k;
    p.v_new = v;
    p.slot_mapping = slot_mapping;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.counters = counters;
    dim3 grid(shp->num_seqs, shp->num_kv_heads, max_num_partitions);
    e = launch(pa::kModeStep, shp, ck, tmk, tmv, p, grid, stream);
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

// CTAs of the balanced step's grid on the current device: one wave, every SM
// holding the decode kernel's resident CTAs.
cudaError_t balanced_grid(int* num_ctas, bool fp8) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    *num_ctas = sms * (fp8 ? pa::kMinCtasPerSmFp8 : pa::kMinCtasPerSm);
    return cudaSuccess;
}

// Consumer warps of the larger of the two grids (16-bit and FP8 caches).
cudaError_t balanced_max_warps(int* warps) {
    int a = 0, b = 0;
    cudaError_t e = balanced_grid(&a, false);
    if (e == cudaSuccess) e = balanced_grid(&b, true);
    if (e != cudaSuccess) return e;
    *warps = (a > b ? a : b) * pa::kConsumerWarps;
    return cudaSuccess;
}

struct BalancedWorkspace {
    int* counters;
    float* rec_m;
    float* rec_l;
    float* rec_o;
    size_t bytes;
};

// [counters B*Hkv][rec_m R*G][rec_l R*G][rec_o R*G*D], each part 256-byte
// aligned, R = max consumer warps + B*Hkv.
BalancedWorkspace balanced_layout(const pa_shape* s, int max_warps, void* base) {
    const size_t B = s->num_seqs, Hkv = s->num_kv_heads, G = s->num_q_heads / s->num_kv_heads;
    const size_t R = (size_t)max_warps + B * Hkv;
    BalancedWorkspace w{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += round256(bytes);
        return static_cast<unsigned char*>(base) + at;
    };
    w.counters = reinterpret_cast<int*>(take(B * Hkv * sizeof(int)));
    w.rec_m = reinterpret_cast<float*>(take(R * G * sizeof(float)));
    w.rec_l = reinterpret_cast<float*>(take(R * G * sizeof(float)));
    w.rec_o = reinterpret_cast<float*>(take(R * G * s->head_dim * sizeof(float)));
    w.bytes = off;
    return w;
}

int decode_step_balanced(const void* q, const void* k, const void* v, const int64_t* slot_mapping,
                         void* k_cache, void* v_cache, const int32_t* block_tables,
                         const int32_t* context_lens, float scale, void* workspace,
                         size_t workspace_bytes, void* out, const pa_shape* shp, void* stream,
                         const CacheKind& ck) {
    int st = check_decode_args(q, k_cache, v_cache, block_tables, context_lens, shp);
    if (st != PA_OK) return st;
    if ((st = check_kind(shp, ck)) != PA_OK) return st;
    if (shp->num_seqs == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !out || !aligned16(k) || !aligned16(v) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PA_ERR_INVALID_ARG;
    if ((int64_t)shp->num_seqs * shp->num_kv_heads * shp->max_blocks_per_seq *
            (shp->block_size / pa::kTileTokens) >= (1ll << 31))
        return PA_ERR_UNSUPPORTED;
    if (!workspace || !aligned16(workspace)) return PA_ERR_WORKSPACE;
    int num_ctas = 0, max_warps = 0;
    cudaError_t e = balanced_grid(&num_ctas, ck.fp8);
    if (e == cudaSuccess) e = balanced_max_warps(&max_warps);
    if (e != cudaSuccess) return cuda_fail(e);
    BalancedWorkspace w = balanced_layout(shp, max_warps, workspace);
    if (w.bytes > workspace_bytes) return PA_ERR_WORKSPACE;
    CUtensorMap tmk, tmv;
    if ((st = encode_cache_map(&tmk, k_cache, shp, ck.fp8)) != PA_OK) return st;
    if ((st = encode_cache_map(&tmv, v_cache, shp, ck.fp8)) != PA_OK) return st;
    int* err = nullptr;
    e = error_word(&err);
    if (e != cudaSuccess) return cuda_fail(e);
    pa::BalancedParams p{};
    p.q = q;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = out;
    p.err = err;
    p.scale_log2 = scale * ck.k_scale * pa::kLog2e;
    p.num_q_heads = shp->num_q_heads;
    p.group = shp->num_q_heads / shp->num_kv_heads;
    p.max_blocks_per_seq = shp->max_blocks_per_seq;
    p.block_size = shp->block_size;
    p.num_blocks = shp->num_blocks;
    p.k_new = k;
    p.v_new = v;
    p.slot_mapping = slot_mapping;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.counters = w.counters;
    p.num_kv_heads = shp->num_kv_heads;
    p.k_scale = ck.k_scale;
    p.v_scale = ck.v_scale;
    p.num_seqs = shp->num_seqs;
    p.num_warps = num_ctas * pa::kConsumerWarps;
    p.rec_o = w.rec_o;
    p.rec_m = w.rec_m;
    p.rec_l = w.rec_l;
    e = pa::launch_balanced(shp->dtype, shp->head_dim, ck.fp8, tmk, tmv, p, num_ctas,
                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

// Whether pa_prefill takes the tcgen05 kernel: head_dim 128, a group of 1, 2,
// 4 or 8, a positive scale, and chunks that can fill its 128 rows.
bool prefill_uses_tc(const pa_shape* shp, float scale, int32_t max_query_len) {
    const int group = shp->num_q_heads / shp->num_kv_heads;
    return pa::prefill_tc_supported(shp->head_dim, group, scale) && max_query_len >= 128 / group;
}

size_t prefill_sched_bytes(const pa_shape* shp, int32_t max_query_len) {
    const int group = shp->num_q_heads / shp->num_kv_heads;
    const size_t n = (size_t)shp->num_seqs * pa::prefill_tc_chunks(group, max_query_len);
    return (n * sizeof(int32_t) + 255) & ~(size_t)255;
}

int prefill_any(const void* q, const void* k_cache, const void* v_cache,
                const int32_t* block_tables, const int32_t* context_lens,
                const int32_t* query_start, float scale, int32_t max_query_len, void* workspace,
                size_t workspace_bytes, void* out, const pa_shape* shp, void* stream,
                bool mma_sync_only) {
    int st = check_decode_args(q, k_cache, v_cache, block_tables, context_lens, shp);
    if (st != PA_OK) return st;
    if (max_query_len < 0) return PA_ERR_INVALID_ARG;
    if (shp->num_seqs == 0 || max_query_len == 0) return PA_OK;
    if (!query_start || (reinterpret_cast<uintptr_t>(query_start) & 3u) || !out || !aligned16(out))
        return PA_ERR_INVALID_ARG;
    const int64_t qtiles = (max_query_len + 15) / 16;
    if (qtiles > 0x7fffffffll) return PA_ERR_UNSUPPORTED;
    const bool use_tc = !mma_sync_only && prefill_uses_tc(shp, scale, max_query_len);
    if (use_tc && workspace &&
        (!aligned16(workspace) || workspace_bytes < prefill_sched_bytes(shp, max_query_len)))
        return PA_ERR_INVALID_ARG;
    CUtensorMap tmk, tmv;
    if ((st = encode_cache_map(&tmk, k_cache, shp, false)) != PA_OK) return st;
    if ((st = encode_cache_map(&tmv, v_cache, shp, false)) != PA_OK) return st;
    int* err = nullptr;
    cudaError_t e = error_word(&err);
    if (e != cudaSuccess) return cuda_fail(e);
    pa::PrefillParams p{};
    p.q = q;
    p.out = out;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.query_start = query_start;
    p.err = err;
    p.scale_log2 = scale * pa::kLog2e;
    p.num_q_heads = shp->num_q_heads;
    p.group = shp->num_q_heads / shp->num_kv_heads;
    p.max_blocks_per_seq = shp->max_blocks_per_seq;
    p.block_size = shp->block_size;
    p.num_blocks = shp->num_blocks;
    // the tcgen05 kernel's 128-row tiles pay off once a chunk can fill one
    if (use_tc) {
        p.max_chunks = pa::prefill_tc_chunks(p.group, max_query_len);
        p.num_seqs = shp->num_seqs;
        if ((int64_t)p.num_seqs * p.max_chunks * shp->num_kv_heads > 0x7fffffffll)
            return PA_ERR_UNSUPPORTED;
        const cudaStream_t st_ = static_cast<cudaStream_t>(stream);
        if (workspace) {
            int32_t* sched = static_cast<int32_t*>(workspace);
            e = pa::launch_prefill_tc_plan(p, sched, st_);
            p.sched = sched;
        }
        if (e == cudaSuccess) e = pa::launch_prefill_tc(shp->dtype, tmk, tmv, p, shp->num_kv_heads, st_);
    } else {
        dim3 grid((unsigned)qtiles, shp->num_kv_heads, shp->num_seqs);
        e = pa::launch_prefill(shp->dtype, shp->head_dim, tmk, tmv, p, grid,
                               static_cast<cudaStream_t>(stream));
    }
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

size_t pa_balanced_workspace_size(const pa_shape* shp) {
    if (check_shape(shp, true) != PA_OK) return 0;
    int max_warps = 0;
    if (balanced_max_warps(&max_warps) != cudaSuccess) return 0;
    return balanced_layout(shp, max_warps, nullptr).bytes;
}

int pa_decode_step_balanced(const void* q, const void* k, const void* v,
                            const int64_t* slot_mapping, void* k_cache, void* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens, float scale,
                            void* workspace, size_t workspace_bytes, void* out,
                            const pa_shape* shp, void* stream) {
    return decode_step_balanced(q, k, v, slot_mapping, k_cache, v_cache, block_tables,
                                context_lens, scale, workspace, workspace_bytes, out, shp, stream,
                                kCache16);
}

int pa_decode_step_balanced_fp8(const void* q, const void* k, const void* v,
                                const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens,
                                float scale, float k_scale, float v_scale, void* workspace,
                                size_t workspace_bytes, void* out, const pa_shape* shp,
                                void* stream) {
    return decode_step_balanced(q, k, v, slot_mapping, k_cache, v_cache, block_tables,
                                context_lens, scale, workspace, workspace_bytes, out, shp, stream,
                                CacheKind{true, k_scale, v_scale});
}

int pa_decode(const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, const int32_t* context_lens, float scale,
              void* out, const pa_shape* shp, void* stream) {
    return decode_single(q, k_cache, v_cache, block_tables, context_lens, scale, out, shp,
                         stream, kCache16);
}

size_t pa_split_workspace_size(const pa_shape* shp, int32_t max_context_len,
                               int32_t partition_size) {
    if (check_shape(shp, true) != PA_OK) return 0;
    if (max_context_len < 0 || partition_size <= 0 || partition_size % shp->block_size != 0)
        return 0;
    const size_t parts = (size_t)((max_context_len + partition_size - 1) / partition_size);
    const size_t rows = (size_t)shp->num_seqs * shp->num_q_heads * (parts ? parts : 1);
    return round256(rows * shp->head_dim * sizeof(float)) + 2 * round256(rows * sizeof(float));
}

int pa_decode_split(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, const int32_t* context_lens, float scale,
                    int32_t partition_size, int32_t max_num_partitions, float* tmp_out,
                    float* max_logits, float* exp_sums, const pa_shape* shp, void* stream) {
    return decode_split(q, k_cache, v_cache, block_tables, context_lens, scale, partition_size,
                        max_num_partitions, tmp_out, max_logits, exp_sums, shp, stream,
                        kCache16);
}

int pa_decode_step(const void* q, const void* k, const void* v, const int64_t* slot_mapping,
                   void* k_cache, void* v_cache, const int32_t* block_tables,
                   const int32_t* context_lens, float scale, int32_t partition_size,
                   int32_t max_num_partitions, float* tmp_out, float* max_logits,
                   float* exp_sums, int32_t* counters, void* out, const pa_shape* shp,
                   void* stream) {
    return decode_step(q, k, v, slot_mapping, k_cache, v_cache, block_tables, context_lens, scale,
                       partition_size, max_num_partitions, tmp_out, max_logits, exp_sums,
                       counters, out, shp, stream, kCache16);
}

int pa_reshape_and_cache_fp8(const void* k, const void* v, const int64_t* slot_mapping,
                             void* k_cache, void* v_cache, int64_t num_tokens, float k_scale,
                             float v_scale, const pa_shape* shp, void* stream) {
    int st = check_shape(shp, false);
    if (st != PA_OK) return st;
    if ((st = check_kind(shp, CacheKind{true, k_scale, v_scale})) != PA_OK) return st;
    if (num_tokens < 0 || num_tokens > 0x7fffffffll) return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PA_ERR_INVALID_ARG;
    int* err = nullptr;
    cudaError_t e = error_word(&err);
    if (e != cudaSuccess) return cuda_fail(e);
    e = pa::launch_reshape_and_cache_fp8(shp->dtype, k, v, slot_mapping, k_cache, v_cache,
                                         num_tokens, shp->num_blocks * shp->block_size,
                                         shp->num_kv_heads * shp->head_dim, k_scale, v_scale,
                                         err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int pa_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens, float scale,
                  float k_scale, float v_scale, void* out, const pa_shape* shp, void* stream) {
    return decode_single(q, k_cache, v_cache, block_tables, context_lens, scale, out, shp,
                         stream, CacheKind{true, k_scale, v_scale});
}

int pa_decode_split_fp8(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, const int32_t* context_lens, float scale,
                        float k_scale, float v_scale, int32_t partition_size,
                        int32_t max_num_partitions, float* tmp_out, float* max_logits,
                        float* exp_sums, const pa_shape* shp, void* stream) {
    return decode_split(q, k_cache, v_cache, block_tables, context_lens, scale, partition_size,
                        max_num_partitions, tmp_out, max_logits, exp_sums, shp, stream,
                        CacheKind{true, k_scale, v_scale});
}

int pa_decode_step_fp8(const void* q, const void* k, const void* v, const int64_t* slot_mapping,
                       void* k_cache, void* v_cache, const int32_t* block_tables,
                       const int32_t* context_lens, float scale, float k_scale, float v_scale,
                       int32_t partition_size, int32_t max_num_partitions, float* tmp_out,
                       float* max_logits, float* exp_sums, int32_t* counters, void* out,
                       const pa_shape* shp, void* stream) {
    return decode_step(q, k, v, slot_mapping, k_cache, v_cache, block_tables, context_lens, scale,
                       partition_size, max_num_partitions, tmp_out, max_logits, exp_sums,
                       counters, out, shp, stream, CacheKind{true, k_scale, v_scale});
}

int pa_prefill(const void* q, const void* k_cache, const void* v_cache,
               const int32_t* block_tables, const int32_t* context_lens,
               const int32_t* query_start, float scale, int32_t max_query_len, void* out,
               const pa_shape* shp, void* stream) {
    return prefill_any(q, k_cache, v_cache, block_tables, context_lens, query_start, scale,
                       max_query_len, nullptr, 0, out, shp, stream, false);
}

size_t pa_prefill_workspace_size(const pa_shape* shp, int32_t max_query_len) {
    if (!shp || shp->num_seqs <= 0 || shp->num_kv_heads <= 0 || max_query_len <= 0 ||
        shp->num_q_heads % shp->num_kv_heads != 0)
        return 0;
    // the ordering is only used by the tcgen05 kernel; its scale test is on sign
    return prefill_uses_tc(shp, 1.f, max_query_len) ? prefill_sched_bytes(shp, max_query_len) : 0;
}

int pa_prefill_ws(const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens,
                  const int32_t* query_start, float scale, int32_t max_query_len,
                  void* workspace, size_t workspace_bytes, void* out, const pa_shape* shp,
                  void* stream) {
    return prefill_any(q, k_cache, v_cache, block_tables, context_lens, query_start, scale,
                       max_query_len, workspace, workspace_bytes, out, shp, stream, false);
}

int pa_prefill_mma(const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* block_tables, const int32_t* context_lens,
                   const int32_t* query_start, float scale, int32_t max_query_len, void* out,
                   const pa_shape* shp, void* stream) {
    return prefill_any(q, k_cache, v_cache, block_tables, context_lens, query_start, scale,
                       max_query_len, nullptr, 0, out, shp, stream, true);
}

int pa_copy_async(void* dst, const void* src, size_t nbytes, void* stream) {
    if (nbytes == 0) return PA_OK;
    if (!dst || !src || !aligned16(dst) || !aligned16(src) || (nbytes & 15u))
        return PA_ERR_INVALID_ARG;
    const cudaError_t e = pa::launch_copy16(dst, src, nbytes / 16, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int pa_copy_blocks(const void* k_src, const void* v_src, int64_t src_num_blocks, void* k_dst,
                   void* v_dst, int64_t dst_num_blocks, const int64_t* block_mapping,
                   int64_t num_pairs, const pa_shape* shp, void* stream) {
    int st = check_shape(shp, false);
    if (st != PA_OK) return st;
    if (num_pairs < 0 || num_pairs > 65535 || src_num_blocks <= 0 || dst_num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_pairs == 0) return PA_OK;
    if (!k_src || !v_src || !k_dst || !v_dst || !block_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_src) || !aligned16(v_src) || !aligned16(k_dst) || !aligned16(v_dst) ||
        (reinterpret_cast<uintptr_t>(block_mapping) & 7u))
        return PA_ERR_INVALID_ARG;
    int* err = nullptr;
    cudaError_t e = error_word(&err);
    if (e != cudaSuccess) return cuda_fail(e);
    const int64_t block_bytes =
        (int64_t)shp->block_size * shp->num_kv_heads * shp->head_dim * 2;
    e = pa::launch_copy_blocks(k_src, v_src, src_num_blocks, k_dst, v_dst, dst_num_blocks,
                               block_mapping, num_pairs, block_bytes, err,
                               static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int pa_reduce(const float* tmp_out, const float* max_logits, const float* exp_sums,
              const int32_t* context_lens, int32_t partition_size, int32_t max_num_partitions,
              void* out, const pa_shape* shp, void* stream) {
    int st = check_shape(shp, true);
    if (st != PA_OK) return st;
    if (partition_size <= 0 || partition_size % shp->block_size != 0) return PA_ERR_INVALID_ARG;
    if (max_num_partitions <= 0) return PA_ERR_WORKSPACE;
    if (shp->num_seqs == 0) return PA_OK;
    if (!tmp_out || !max_logits || !exp_sums) return PA_ERR_WORKSPACE;
    if (!context_lens || !out || !aligned16(out) || !aligned16(tmp_out)) return PA_ERR_INVALID_ARG;
    int* err = nullptr;
    cudaError_t e = error_word(&err);
    if (e != cudaSuccess) return cuda_fail(e);
    pa::ReduceParams p{};
    p.tmp_out = tmp_out;
    p.max_logits = max_logits;
    p.exp_sums = exp_sums;
    p.context_lens = context_lens;
    p.out = out;
    p.err = err;
    p.num_q_heads = shp->num_q_heads;
    p.partition_tokens = partition_size;
    p.max_parts = max_num_partitions;
    p.max_context = shp->max_blocks_per_seq * shp->block_size;
    e = pa::launch_reduce(shp->dtype, shp->head_dim, p, shp->num_seqs,
                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

}  // extern "C"
