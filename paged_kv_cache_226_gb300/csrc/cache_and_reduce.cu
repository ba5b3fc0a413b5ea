// reshape_and_cache (the cache write of a decode step) and the log-sum-exp
// merge of the context split.
#include "pa_device.cuh"

namespace pa {

cudaError_t launch_decode_f16(int, int, const CUtensorMap&, const CUtensorMap&,
                              const DecodeParams&, dim3, cudaStream_t);
cudaError_t launch_decode_bf16(int, int, const CUtensorMap&, const CUtensorMap&,
                               const DecodeParams&, dim3, cudaStream_t);

cudaError_t launch_decode_fp8_f16(int, const CUtensorMap&, const CUtensorMap&,
                                  const DecodeParams&, dim3, cudaStream_t);
cudaError_t launch_decode_fp8_bf16(int, const CUtensorMap&, const CUtensorMap&,
                                   const DecodeParams&, dim3, cudaStream_t);

cudaError_t launch_decode_fp8(int dtype, int mode, const CUtensorMap& tmk,
                              const CUtensorMap& tmv, const DecodeParams& p, dim3 grid,
                              cudaStream_t stream) {
    if (dtype == PA_BF16) return launch_decode_fp8_bf16(mode, tmk, tmv, p, grid, stream);
    return launch_decode_fp8_f16(mode, tmk, tmv, p, grid, stream);
}

cudaError_t launch_decode(int dtype, int head_dim, int mode, const CUtensorMap& tmk,
                          const CUtensorMap& tmv, const DecodeParams& p, dim3 grid,
                          cudaStream_t stream) {
    if (dtype == PA_BF16) return launch_decode_bf16(head_dim, mode, tmk, tmv, p, grid, stream);
    return launch_decode_f16(head_dim, mode, tmk, tmv, p, grid, stream);
}

// ---------------------------------------------------------------------------
// reshape_and_cache
// ---------------------------------------------------------------------------
//
// With the cache laid out [num_blocks][block_size][Hkv][D], slot
// s = block * block_size + offset addresses row s of the [num_slots][Hkv*D]
// view, so writing token t is one contiguous row copy (youngju.dev
// "vLLM inference optimization", PagedAttentionManager.append_token writes
// k_cache[last_block, slot_in_block]).  One CTA per token, 16-byte vectors.
__global__ void __launch_bounds__(256)
    reshape_and_cache_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                             const int64_t* __restrict__ slots, uint4* __restrict__ kc,
                             uint4* __restrict__ vc, int64_t num_slots, int vec_per_row,
                             int* err) {
    grid_dependency_wait();
    allow_dependent_launch();
    const int64_t t = blockIdx.x;
    const int64_t s = slots[t];
    if (s < 0) return;                                  // padding token
    if (s >= num_slots) {
        if (threadIdx.x == 0) flag_error(err, PA_DEVERR_BAD_SLOT);
        return;
    }
    const uint4* ks = k + t * vec_per_row;
    const uint4* vs = v + t * vec_per_row;
    uint4* kd = kc + s * vec_per_row;
    uint4* vd = vc + s * vec_per_row;
    for (int i = threadIdx.x; i < vec_per_row; i += blockDim.x) {
        kd[i] = __ldg(ks + i);
        vd[i] = __ldg(vs + i);
    }
}

cudaError_t launch_reshape_and_cache(const void* k, const void* v, const int64_t* slots,
                                     void* kc, void* vc, int64_t num_tokens,
                                     int64_t num_slots, int row_bytes, int* err,
                                     cudaStream_t stream) {
    const int vec = row_bytes / 16;
    int threads = vec < 256 ? ((vec + 31) / 32) * 32 : 256;
    return launch_with_pdl(reshape_and_cache_kernel, dim3((unsigned)num_tokens), dim3(threads), 0,
                           stream, static_cast<const uint4*>(k), static_cast<const uint4*>(v),
                           slots, static_cast<uint4*>(kc), static_cast<uint4*>(vc), num_slots,
                           vec, err);
}

// FP8 cache write: every element becomes the E4M3 code of x / scale (the
// quotient in fp32, round to nearest even, saturating at +-448).  One CTA per
// token; each thread converts 8 elements (16 bytes in, 8 bytes out).
template <typename T>
__global__ void __launch_bounds__(256)
    reshape_and_cache_fp8_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                 const int64_t* __restrict__ slots, uint2* __restrict__ kc,
                                 uint2* __restrict__ vc, int64_t num_slots, int chunks_per_row,
                                 float k_scale, float v_scale, int* err) {
    grid_dependency_wait();
    allow_dependent_launch();
    const int64_t t = blockIdx.x;
    const int64_t s = slots[t];
    if (s < 0) return;
    if (s >= num_slots) {
        if (threadIdx.x == 0) flag_error(err, PA_DEVERR_BAD_SLOT);
        return;
    }
    for (int i = threadIdx.x; i < 2 * chunks_per_row; i += blockDim.x) {
        const bool is_k = i < chunks_per_row;
        const int c = is_k ? i : i - chunks_per_row;
        const float sc = is_k ? k_scale : v_scale;
        const uint4 val = __ldg((is_k ? k : v) + t * chunks_per_row + c);
        const uint32_t w[4] = {val.x, val.y, val.z, val.w};
        uint32_t q[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = Mma<T>::unpack(w[j]);
            q[j] = f32x2_to_e4m3x2(__fdiv_rn(f.y, sc), __fdiv_rn(f.x, sc));
        }
        (is_k ? kc : vc)[s * chunks_per_row + c] = make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
    }
}

cudaError_t launch_reshape_and_cache_fp8(int dtype, const void* k, const void* v,
                                         const int64_t* slots, void* kc, void* vc,
                                         int64_t num_tokens, int64_t num_slots, int row_elems,
                                         float k_scale, float v_scale, int* err,
                                         cudaStream_t stream) {
    const int chunks = row_elems / 8;
    const int threads = 2 * chunks < 256 ? ((2 * chunks + 31) / 32) * 32 : 256;
    const dim3 grid((unsigned)num_tokens);
    if (dtype == PA_BF16)
        return launch_with_pdl(reshape_and_cache_fp8_kernel<__nv_bfloat16>, grid, dim3(threads), 0,
                               stream, static_cast<const uint4*>(k), static_cast<const uint4*>(v),
                               slots, static_cast<uint2*>(kc), static_cast<uint2*>(vc), num_slots,
                               chunks, k_scale, v_scale, err);
    return launch_with_pdl(reshape_and_cache_fp8_kernel<__half>, grid, dim3(threads), 0, stream,
                           static_cast<const uint4*>(k), static_cast<const uint4*>(v), slots,
                           static_cast<uint2*>(kc), static_cast<uint2*>(vc), num_slots, chunks,
                           k_scale, v_scale, err);
}

// ---------------------------------------------------------------------------
// log-sum-exp merge
// ---------------------------------------------------------------------------
//
// For (b, h): S = min(ceil(L/P), max_parts) partitions with normalised
// outputs o_s, maxima m_s and sums l_s.  M = max m_s, w_s = l_s e^(m_s - M),
// out = sum w_s o_s / sum w_s.  One CTA of 8 warps per (b, h): the warps take
// the partitions round robin (lane l owns dims [D/32 * l, D/32 * (l+1))),
// two partitions in flight per warp, then merge through shared memory.
constexpr int kReduceWarps = 8;

template <int V>
__device__ __forceinline__ void load_floats(const float* p, float (&x)[V]) {
    if constexpr (V == 4) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p));
        x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w;
    } else {
        const float2 a = __ldg(reinterpret_cast<const float2*>(p));
        x[0] = a.x, x[1] = a.y;
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kReduceWarps * 32)
    lse_reduce_kernel(const __grid_constant__ ReduceParams p) {
    constexpr int V = D / 32;                       // floats per lane (4 or 2)
    __shared__ float red_o[kReduceWarps][D];
    __shared__ float red_l[kReduceWarps];
    __shared__ float red_m[kReduceWarps];
    grid_dependency_wait();
    allow_dependent_launch();
    const int h = blockIdx.x;
    const int b = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int L = p.context_lens[b];
    if (L < 0 || L > p.max_context) {
        if (tid == 0 && h == 0) flag_error(p.err, PA_DEVERR_BAD_CONTEXT);
        L = L < 0 ? 0 : p.max_context;
    }
    int S = (L + p.partition_tokens - 1) / p.partition_tokens;
    S = min(S, p.max_parts);
    T* out = reinterpret_cast<T*>(p.out) + ((size_t)b * p.num_q_heads + h) * D;
    if (S <= 0) {
        for (int d = tid; d < D; d += blockDim.x) out[d] = from_float<T>(0.f);
        return;
    }
    const size_t base = ((size_t)b * p.num_q_heads + h) * p.max_parts;
    const float* ml = p.max_logits + base;
    const float* es = p.exp_sums + base;
    const float* o = p.tmp_out + base * D + lane * V;

    // M = max_s m_s
    float m = -INFINITY;
    for (int s = tid; s < S; s += blockDim.x) m = fmaxf(m, __ldg(ml + s));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) red_m[warp] = m;
    __syncthreads();
    float M = red_m[0];
#pragma unroll
    for (int w = 1; w < kReduceWarps; ++w) M = fmaxf(M, red_m[w]);

    float acc[V];
#pragma unroll
    for (int i = 0; i < V; ++i) acc[i] = 0.f;
    float den = 0.f;
    int s = warp;
    for (; s + kReduceWarps < S; s += 2 * kReduceWarps) {
        const int s2 = s + kReduceWarps;
        const float w0 = __ldg(es + s) * __expf(__ldg(ml + s) - M);
        const float w1 = __ldg(es + s2) * __expf(__ldg(ml + s2) - M);
        float x0[V], x1[V];
        load_floats<V>(o + (size_t)s * D, x0);
        load_floats<V>(o + (size_t)s2 * D, x1);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] += w0 * x0[i] + w1 * x1[i];
        den += w0 + w1;
    }
    if (s < S) {
        const float w0 = __ldg(es + s) * __expf(__ldg(ml + s) - M);
        float x0[V];
        load_floats<V>(o + (size_t)s * D, x0);
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] += w0 * x0[i];
        den += w0;
    }
#pragma unroll
    for (int i = 0; i < V; ++i) red_o[warp][lane * V + i] = acc[i];
    if (lane == 0) red_l[warp] = den;
    __syncthreads();
    for (int d = tid; d < D; d += blockDim.x) {
        float num = 0.f, dd = 0.f;
#pragma unroll
        for (int w = 0; w < kReduceWarps; ++w) {
            num += red_o[w][d];
            dd += red_l[w];
        }
        out[d] = from_float<T>(num / dd);
    }
}

cudaError_t launch_reduce(int dtype, int head_dim, const ReduceParams& p, int num_seqs,
                          cudaStream_t stream) {
    dim3 grid(p.num_q_heads, num_seqs);
    const dim3 threads(kReduceWarps * 32);
    if (dtype == PA_BF16) {
        if (head_dim == 64)
            return launch_with_pdl(lse_reduce_kernel<__nv_bfloat16, 64>, grid, threads, 0, stream, p);
        return launch_with_pdl(lse_reduce_kernel<__nv_bfloat16, 128>, grid, threads, 0, stream, p);
    }
    if (head_dim == 64)
        return launch_with_pdl(lse_reduce_kernel<__half, 64>, grid, threads, 0, stream, p);
    return launch_with_pdl(lse_reduce_kernel<__half, 128>, grid, threads, 0, stream, p);
}

}  // namespace pa
