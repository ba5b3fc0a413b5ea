// reshape_and_cache (the cache write of a decode step) and the log-sum-exp
// merge of the context split.
#include "pa_device.cuh"

namespace pa {

cudaError_t launch_decode_f16(int, bool, const CUtensorMap&, const CUtensorMap&,
                              const DecodeParams&, dim3, cudaStream_t);
cudaError_t launch_decode_bf16(int, bool, const CUtensorMap&, const CUtensorMap&,
                               const DecodeParams&, dim3, cudaStream_t);

cudaError_t launch_decode(int dtype, int head_dim, bool split, const CUtensorMap& tmk,
                          const CUtensorMap& tmv, const DecodeParams& p, dim3 grid,
                          cudaStream_t stream) {
    if (dtype == PA_BF16) return launch_decode_bf16(head_dim, split, tmk, tmv, p, grid, stream);
    return launch_decode_f16(head_dim, split, tmk, tmv, p, grid, stream);
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
    reshape_and_cache_kernel<<<dim3((unsigned)num_tokens), threads, 0, stream>>>(
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), slots,
        static_cast<uint4*>(kc), static_cast<uint4*>(vc), num_slots, vec, err);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// log-sum-exp merge
// ---------------------------------------------------------------------------
//
// For (b, h): S = min(ceil(L/P), max_parts) partitions with normalised
// outputs o_s, maxima m_s and sums l_s.  M = max m_s, w_s = l_s e^(m_s - M),
// out = sum w_s o_s / sum w_s.  One CTA of D threads per (b, h); thread d
// owns output dim d; the m_s / l_s reads are warp-broadcast.
template <typename T, int D>
__global__ void __launch_bounds__(D) lse_reduce_kernel(const __grid_constant__ ReduceParams p) {
    const int h = blockIdx.x;
    const int b = blockIdx.y;
    const int d = threadIdx.x;
    int L = p.context_lens[b];
    if (L < 0 || L > p.max_context) {
        if (d == 0 && h == 0) flag_error(p.err, PA_DEVERR_BAD_CONTEXT);
        L = L < 0 ? 0 : p.max_context;
    }
    int S = (L + p.partition_tokens - 1) / p.partition_tokens;
    S = min(S, p.max_parts);
    T* out = reinterpret_cast<T*>(p.out) + ((size_t)b * p.num_q_heads + h) * D;
    if (S <= 0) {
        out[d] = from_float<T>(0.f);
        return;
    }
    const size_t base = ((size_t)b * p.num_q_heads + h) * p.max_parts;
    const float* ml = p.max_logits + base;
    const float* es = p.exp_sums + base;
    const float* o = p.tmp_out + base * D + d;
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, __ldg(ml + s));
    float num = 0.f, den = 0.f;
    int s = 0;
    for (; s + 4 <= S; s += 4) {
        const float w0 = __ldg(es + s) * __expf(__ldg(ml + s) - M);
        const float w1 = __ldg(es + s + 1) * __expf(__ldg(ml + s + 1) - M);
        const float w2 = __ldg(es + s + 2) * __expf(__ldg(ml + s + 2) - M);
        const float w3 = __ldg(es + s + 3) * __expf(__ldg(ml + s + 3) - M);
        num += w0 * __ldg(o + (size_t)s * D) + w1 * __ldg(o + (size_t)(s + 1) * D) +
               w2 * __ldg(o + (size_t)(s + 2) * D) + w3 * __ldg(o + (size_t)(s + 3) * D);
        den += (w0 + w1) + (w2 + w3);
    }
    for (; s < S; ++s) {
        const float w = __ldg(es + s) * __expf(__ldg(ml + s) - M);
        num += w * __ldg(o + (size_t)s * D);
        den += w;
    }
    out[d] = from_float<T>(num / den);
}

cudaError_t launch_reduce(int dtype, int head_dim, const ReduceParams& p, int num_seqs,
                          cudaStream_t stream) {
    dim3 grid(p.num_q_heads, num_seqs);
    if (dtype == PA_BF16) {
        if (head_dim == 64)
            lse_reduce_kernel<__nv_bfloat16, 64><<<grid, 64, 0, stream>>>(p);
        else
            lse_reduce_kernel<__nv_bfloat16, 128><<<grid, 128, 0, stream>>>(p);
    } else {
        if (head_dim == 64)
            lse_reduce_kernel<__half, 64><<<grid, 64, 0, stream>>>(p);
        else
            lse_reduce_kernel<__half, 128><<<grid, 128, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace pa
