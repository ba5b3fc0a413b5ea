// Paged prefill / chunked-prefill attention: every new token of a sequence
// attends causally over the sequence's cache through its block table.
//
// Sequence b holds L_b tokens, the last C_b of which are new (their K/V were
// written by reshape_and_cache): new token i sits at position
// p = L_b - C_b + i and attends to positions 0..p (ta-paperlens page,
// prefill vs decode; techfeed summary, chunked prefill).  One CTA serves 16
// new tokens of one (sequence, KV head): consumer warp w computes query head
// g*G + w for those 16 tokens (16 rows of an m16n8k16 product), all warps
// share each K/V tile that a producer warp streams through the TMA ring.
// Per tile and warp: S = Q K^T (16 x 16 over D), causal mask, fp32 online
// softmax per row, O += P V with P rounded to the 16-bit type (bf16: hi +
// lo parts), P reused straight from the score fragments.
#include "decode_tile.cuh"
#include "prefill_internal.h"

namespace pa {

constexpr int kPrefillTileTokens = 16;     // query tokens per CTA
constexpr int kPrefillStages = 4;

template <int D>
struct PrefillLayout {
    static constexpr int kHalves = D / kBoxElems;
    static constexpr int kTileBytes = kHalves * kBox16Bytes;      // K or V of 16 tokens
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kDynamicSmem = kPrefillStages * kStageBytes + 1024;
};

template <typename T, int D>
__global__ void __launch_bounds__((kMaxGroup + 1) * 32)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v,
                         const __grid_constant__ PrefillParams p) {
    using Lay = PrefillLayout<D>;
    using M = Mma<T>;
    constexpr int kKSteps = D / 16;
    constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;
    __shared__ __align__(8) uint64_t full_bar[kPrefillStages];
    __shared__ __align__(8) uint64_t empty_bar[kPrefillStages];
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int qt = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group;

    grid_dependency_wait();
    allow_dependent_launch();
    const int max_ctx = p.max_blocks_per_seq * p.block_size;
    int L = p.context_lens[b];
    if (L < 0 || L > max_ctx) {
        if (threadIdx.x == 0 && qt == 0 && g == 0) flag_error(p.err, PA_DEVERR_BAD_CONTEXT);
        L = L < 0 ? 0 : max_ctx;
    }
    const int q0 = p.query_start[b];
    int C = p.query_start[b + 1] - q0;
    if (C > L) {
        if (threadIdx.x == 0 && qt == 0 && g == 0) flag_error(p.err, PA_DEVERR_BAD_CONTEXT);
        C = L;
    }
    const int t0 = qt * kPrefillTileTokens;                 // first new token of the CTA
    if (t0 >= C) return;
    const int rows = min(kPrefillTileTokens, C - t0);
    const int last_pos = L - C + t0 + rows - 1;             // the last token's position
    const int n_tiles = last_pos / kTileTokens + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPrefillStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], G);                    // every consumer warp reads a tile
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == G) {
        // producer: block table -> TMA boxes, tiles 0 .. n_tiles - 1
        if (lane == 0) {
            prefetch_tensor_map(&tmap_k);
            prefetch_tensor_map(&tmap_v);
        }
        const int32_t* table = p.block_tables + (size_t)b * p.max_blocks_per_seq;
        const int tiles_per_block = p.block_size / kTileTokens;
        bool ok = true;
        for (int i0 = 0; i0 < n_tiles && ok; i0 += 32) {
            int blk = 0;
            if (i0 + lane < n_tiles) {
                blk = __ldg(table + (i0 + lane) / tiles_per_block);
                if (blk < 0 || blk >= p.num_blocks) flag_error(p.err, PA_DEVERR_BAD_CONTEXT);
            }
            const int cnt = min(32, n_tiles - i0);
            for (int k = 0; k < cnt; ++k) {
                const int pblk = __shfl_sync(0xffffffffu, blk, k);
                if (lane == 0) {
                    const int it = i0 + k;
                    const int st = it % kPrefillStages;
                    if (it >= kPrefillStages &&
                        !mbar_wait(&empty_bar[st], ((it / kPrefillStages) - 1) & 1)) {
                        flag_error(p.err, PA_DEVERR_WAIT_TIMEOUT);
                        ok = false;
                    } else {
                        mbar_arrive_expect_tx(&full_bar[st], Lay::kStageBytes);
                        const int sub = (it % tiles_per_block) * kTileTokens;
                        uint8_t* kdst = smem + st * Lay::kStageBytes;
                        uint8_t* vdst = kdst + Lay::kTileBytes;
#pragma unroll
                        for (int hh = 0; hh < Lay::kHalves; ++hh) {
                            tma_load_4d(kdst + hh * kBox16Bytes, &tmap_k, &full_bar[st],
                                        hh * kBoxElems, g, sub, pblk);
                            tma_load_4d(vdst + hh * kBox16Bytes, &tmap_v, &full_bar[st],
                                        hh * kBoxElems, g, sub, pblk);
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
            }
        }
        return;
    }

    // ----------------------------------------------------------------------
    // consumer warp: query head h = g*G + warp for new tokens t0 .. t0+15
    // (rows r8 and r8+8 of this lane; columns 2c4, 2c4+1 of each 8-wide tile)
    // ----------------------------------------------------------------------
    const int r8 = lane >> 2, c4 = lane & 3;
    const int h = g * G + warp;
    // Q as the A operand (16 tokens x 16 dims per k-step); rows past the chunk are zero
    uint32_t qa[kKSteps][4];
    {
        const T* qlo = reinterpret_cast<const T*>(p.q) +
                       ((size_t)(q0 + t0 + min(r8, rows - 1)) * p.num_q_heads + h) * D;
        const T* qhi = reinterpret_cast<const T*>(p.q) +
                       ((size_t)(q0 + t0 + min(r8 + 8, rows - 1)) * p.num_q_heads + h) * D;
        const bool vlo = r8 < rows, vhi = r8 + 8 < rows;
#pragma unroll
        for (int kk = 0; kk < kKSteps; ++kk) {
            const int d = kk * 16 + 2 * c4;
            qa[kk][0] = vlo ? __ldg(reinterpret_cast<const uint32_t*>(qlo + d)) : 0u;
            qa[kk][1] = vhi ? __ldg(reinterpret_cast<const uint32_t*>(qhi + d)) : 0u;
            qa[kk][2] = vlo ? __ldg(reinterpret_cast<const uint32_t*>(qlo + d + 8)) : 0u;
            qa[kk][3] = vhi ? __ldg(reinterpret_cast<const uint32_t*>(qhi + d + 8)) : 0u;
        }
    }
    float o[kKSteps * 2][4];                 // O: 16 rows x D, 8-dim column tiles
#pragma unroll
    for (int n = 0; n < kKSteps * 2; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY;    // reference max of rows r8, r8+8 (log2)
    float l0 = 0.f, l1 = 0.f;                // this lane's share of their sums
    // causal limits of rows r8, r8+8 (inclusive); rows past the chunk are
    // clamped to the context (their outputs are not written)
    const int pos0 = min(L - C + t0 + r8, L - 1);
    const int pos1 = min(L - C + t0 + r8 + 8, L - 1);
    // ldmatrix rows: K as B operand (no transpose): matrices (tok 0-7, lo), (tok 0-7, hi),
    // (tok 8-15, lo), (tok 8-15, hi); V as B operand (transposed): (tok 0-7, d0),
    // (tok 8-15, d0), (tok 0-7, d0+8), (tok 8-15, d0+8)
    const int k_tok = ((lane >> 4) << 3) + (lane & 7);
    const int k_hi = (lane >> 3) & 1;
    const int v_tok = (((lane >> 3) & 1) << 3) + (lane & 7);
    const int v_hi = lane >> 4;

    for (int it = 0; it < n_tiles; ++it) {
        const int st = it % kPrefillStages;
        bool ok = mbar_wait(&full_bar[st], (it / kPrefillStages) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) flag_error(p.err, PA_DEVERR_WAIT_TIMEOUT);
            return;
        }
        const uint32_t kbase = smem_u32(smem + st * Lay::kStageBytes);
        const uint32_t vbase = kbase + Lay::kTileBytes;
        // S = Q K^T: tokens 0-7 (s0) and 8-15 (s1) of the tile
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < kKSteps; ++kk) {
            const int chunk = 2 * kk + k_hi;
            const uint32_t addr = kbase + (chunk >> 3) * kBox16Bytes + k_tok * 128 +
                                  (((chunk & 7) ^ (k_tok & 7)) << 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(addr, b0, b1, b2, b3);
            M::run(s0, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
            M::run(s1, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
        }
        // causal mask (position j visible to a row iff j <= its position), log2 units
        const int j0 = it * kTileTokens + 2 * c4;
        float x[8] = {s0[0], s0[1], s1[0], s1[1], s0[2], s0[3], s1[2], s1[3]};
        const int js[4] = {j0, j0 + 1, j0 + 8, j0 + 9};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[e] = js[e] <= pos0 ? x[e] * p.scale_log2 : -INFINITY;          // row r8
            x[4 + e] = js[e] <= pos1 ? x[4 + e] * p.scale_log2 : -INFINITY;  // row r8+8
        }
        float mx0 = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
        float mx1 = fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const bool up0 = mx0 > m0 + kRescaleThresholdLog2;
        const bool up1 = mx1 > m1 + kRescaleThresholdLog2;
        if (__any_sync(0xffffffffu, up0 || up1)) {
            const float n0 = up0 ? mx0 : m0, n1 = up1 ? mx1 : m1;
            const float f0 = ex2(m0 - n0), f1 = ex2(m1 - n1);
#pragma unroll
            for (int n = 0; n < kKSteps * 2; ++n) {
                o[n][0] *= f0;
                o[n][1] *= f0;
                o[n][2] *= f1;
                o[n][3] *= f1;
            }
            l0 *= f0;
            l1 *= f1;
            m0 = n0;
            m1 = n1;
        }
        float e[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            e[i] = ex2(x[i] - m0);
            e[4 + i] = ex2(x[4 + i] - m1);
        }
        // P as the A operand: a0 = (row r8, tok 2c4..), a1 = (row r8+8, ..),
        // a2 = (row r8, tok 8+2c4..), a3 = (row r8+8, tok 8+..)
        const uint32_t pa0 = M::pack(e[0], e[1]), pa1 = M::pack(e[4], e[5]);
        const uint32_t pa2 = M::pack(e[2], e[3]), pa3 = M::pack(e[6], e[7]);
        uint32_t pl0 = 0u, pl1 = 0u, pl2 = 0u, pl3 = 0u;
        if (kSplitP) {
            const float2 u0 = M::unpack(pa0), u1 = M::unpack(pa1);
            const float2 u2 = M::unpack(pa2), u3 = M::unpack(pa3);
            pl0 = M::pack(e[0] - u0.x, e[1] - u0.y);
            pl1 = M::pack(e[4] - u1.x, e[5] - u1.y);
            pl2 = M::pack(e[2] - u2.x, e[3] - u2.y);
            pl3 = M::pack(e[6] - u3.x, e[7] - u3.y);
            l0 += (e[0] + e[1]) + (e[2] + e[3]);
            l1 += (e[4] + e[5]) + (e[6] + e[7]);
        } else {
            const float2 u0 = M::unpack(pa0), u1 = M::unpack(pa1);
            const float2 u2 = M::unpack(pa2), u3 = M::unpack(pa3);
            l0 += (u0.x + u0.y) + (u2.x + u2.y);
            l1 += (u1.x + u1.y) + (u3.x + u3.y);
        }
        // O += P V.  V rows past the context end get P = 0 but may hold stale
        // non-finite bits, so in the last tile their halves of the V
        // fragments are cleared in registers (the tile is shared by all warps
        // and stays untouched).
        const bool tail = (it + 1) * kTileTokens > L;
        const int jt = it * kTileTokens + 2 * c4;          // tokens of fragment b0: jt, jt+1
        const uint32_t keep_lo = (jt < L ? 0x0000ffffu : 0u) | (jt + 1 < L ? 0xffff0000u : 0u);
        const uint32_t keep_hi = (jt + 8 < L ? 0x0000ffffu : 0u) | (jt + 9 < L ? 0xffff0000u : 0u);
#pragma unroll
        for (int np = 0; np < kKSteps; ++np) {
            const int chunk = 2 * np + v_hi;
            const uint32_t addr = vbase + (chunk >> 3) * kBox16Bytes + v_tok * 128 +
                                  (((chunk & 7) ^ (v_tok & 7)) << 4);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(addr, b0, b1, b2, b3);
            if (tail) {
                b0 &= keep_lo;
                b2 &= keep_lo;
                b1 &= keep_hi;
                b3 &= keep_hi;
            }
            M::run(o[2 * np], pa0, pa1, pa2, pa3, b0, b1);
            M::run(o[2 * np + 1], pa0, pa1, pa2, pa3, b2, b3);
            if (kSplitP) {
                M::run(o[2 * np], pl0, pl1, pl2, pl3, b0, b1);
                M::run(o[2 * np + 1], pl0, pl1, pl2, pl3, b2, b3);
            }
        }
        release_stage(&empty_bar[st], lane);
    }

    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float i0 = 1.f / l0, i1 = 1.f / l1;
    T* out0 = reinterpret_cast<T*>(p.out) + ((size_t)(q0 + t0 + r8) * p.num_q_heads + h) * D;
    T* out1 = reinterpret_cast<T*>(p.out) + ((size_t)(q0 + t0 + r8 + 8) * p.num_q_heads + h) * D;
#pragma unroll
    for (int n = 0; n < kKSteps * 2; ++n) {
        const int d = 8 * n + 2 * c4;
        if (r8 < rows) *reinterpret_cast<uint32_t*>(out0 + d) = M::pack(o[n][0] * i0, o[n][1] * i0);
        if (r8 + 8 < rows) *reinterpret_cast<uint32_t*>(out1 + d) = M::pack(o[n][2] * i1, o[n][3] * i1);
    }
}

template <typename T, int D>
cudaError_t launch_prefill_t(const CUtensorMap& tmk, const CUtensorMap& tmv,
                             const PrefillParams& p, dim3 grid, cudaStream_t stream) {
    const int smem = PrefillLayout<D>::kDynamicSmem;
    cudaError_t e = cudaFuncSetAttribute(paged_prefill_kernel<T, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_with_pdl(paged_prefill_kernel<T, D>, grid, dim3((p.group + 1) * 32), smem,
                           stream, tmk, tmv, p);
}

cudaError_t launch_prefill(int dtype, int head_dim, const CUtensorMap& tmk,
                           const CUtensorMap& tmv, const PrefillParams& p, dim3 grid,
                           cudaStream_t stream) {
    if (dtype == PA_BF16) {
        if (head_dim == 64) return launch_prefill_t<__nv_bfloat16, 64>(tmk, tmv, p, grid, stream);
        return launch_prefill_t<__nv_bfloat16, 128>(tmk, tmv, p, grid, stream);
    }
    if (head_dim == 64) return launch_prefill_t<__half, 64>(tmk, tmv, p, grid, stream);
    return launch_prefill_t<__half, 128>(tmk, tmv, p, grid, stream);
}

}  // namespace pa
