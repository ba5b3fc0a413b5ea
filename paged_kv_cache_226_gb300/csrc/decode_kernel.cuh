// Paged decode attention kernel for sm_103a.
//
// One CTA serves one (sequence b, KV head g[, context partition s]) and the
// G = Hq/Hkv query heads that read KV head g.  It walks the sequence's block
// table and gathers K and V while it computes (ta-paperlens "LLM serving
// from scratch", section on fragmentation and PagedAttention).
//
// Data movement: a producer warp reads the block table and issues the TMA
// boxes of each 16-token tile ([16 tokens][64 dims] of one KV head per box,
// 128 B rows, 128 B swizzle; K then V) into a shared-memory ring guarded by
// mbarriers (4 stages of 8 KiB, 8 of 4 KiB for an FP8 cache), two tiles per
// round with one lane per box; a block of 32 tokens is two tiles.  The two
// consumer warps take the tiles round robin (FP8: in pairs); six CTAs per SM.
//
// Math per tile and warp (the G <= 8 query heads of the group are the N = 8
// columns of two m16n8k16 tile products; columns >= G are zero):
//   S^T[t][h] = K[t] . q[h]            one product per 16 dims
//   online softmax in log2 units with a lazily raised running max: the
//   accumulator is rescaled only when a tile's column max exceeds the max in
//   use by more than 2^8, so exp2(s - m) stays below 256 and fp32 is exact
//   enough; the result is identical in exact arithmetic because numerator
//   and denominator share the same reference max;
//   P is rounded to the cache's 16-bit type -- for fp16 once (the row sum l
//   accumulates the rounded values), for bf16 as a hi + lo pair of bf16
//   values whose sum carries P to ~2^-17 -- transposed in registers with
//   movmatrix, and O^T[d][h] += V^T[d][:] . P^T[:][h] with fp32 accumulation.
// The consumer warps' (m, l, O) are merged through shared memory at the end;
// a partitioned CTA writes a record, and in the fused step the last one of
// a (sequence, KV head) merges the records.
#pragma once

#include "decode_tile.cuh"

namespace pa {

template <int D, bool kFp8 = false>
struct DecodeLayout {
    static constexpr int kRing = kFp8 ? kStagesFp8 : kStages;     // tiles in flight per CTA
    // TMA-staged tiles: 16 tokens x (64 dims x 2 B | 128 dims x 1 B) per box
    static constexpr int kHalves = kFp8 ? 1 : D / kBoxElems;      // boxes per staged tile
    static constexpr int kBoxBytes = kTileTokens * 128;            // 2 KB
    static constexpr int kTileBytes = kHalves * kBoxBytes;         // one of K or V
    static constexpr int kStageBytes = 2 * kTileBytes;             // K and V
    static constexpr int kPipeBytes = kRing * kStageBytes;
    // 16-bit compute tiles (the layout ldmatrix reads): D/64 boxes of [16][128 B]
    static constexpr int kHalves16 = D / kBoxElems;
    static constexpr int kTile16Bytes = kHalves16 * kBoxBytes;
    static constexpr int kConvBytes = 0;     // FP8 codes go from the stage to registers
    // merge area: per warp, O[8][D] then m_used[8], l[8], m_true[8]
    static constexpr int kMergeFloatsPerWarp = kMaxGroup * D + 3 * kMaxGroup;
    static constexpr int kMergeBytes = kConsumerWarps * kMergeFloatsPerWarp * 4;
    static constexpr int kBodyBytes = (kPipeBytes + kConvBytes) > kMergeBytes
                                          ? (kPipeBytes + kConvBytes) : kMergeBytes;
    // q^T fragments of the group, [D/16 k-steps][32 lanes][2 words], read
    // per k-step instead of held in 16 registers through the tile loop
    static constexpr int kQBytes = (D / 16) * 32 * 8;
    static constexpr int kDynamicSmem = kBodyBytes + kQBytes + 1024;  // + alignment slack
};

// The fused step's new token, 16-byte chunk c (8 dims) of its K (is_k) or V
// row for KV head g: written to the cache at new_slot and returned as staged
// data: the 16-bit values, or with an FP8 cache the chunk's eight E4M3 codes
// (of x / scale, the quotient in fp32) in .x and .y -- what attention reads
// back from the cache.
template <typename T, int D, bool kFp8>
__device__ __forceinline__ uint4 new_token_chunk(const DecodeParams& p, int b, int g,
                                                 int64_t new_slot, int c, bool is_k) {
    const size_t row = ((size_t)b * p.num_kv_heads + g) * D;
    const uint4 val = __ldg(reinterpret_cast<const uint4*>(
                                reinterpret_cast<const T*>(is_k ? p.k_new : p.v_new) + row) + c);
    const size_t dst = ((size_t)new_slot * p.num_kv_heads + g) * D;
    if (!kFp8) {
        T* cache = reinterpret_cast<T*>(is_k ? p.k_cache : p.v_cache);
        reinterpret_cast<uint4*>(cache + dst)[c] = val;
        return val;
    }
    const float sc = is_k ? p.k_scale : p.v_scale;
    const uint32_t w[4] = {val.x, val.y, val.z, val.w};
    uint16_t q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 f = Mma<T>::unpack(w[j]);
        q[j] = f32x2_to_e4m3x2(__fdiv_rn(f.y, sc), __fdiv_rn(f.x, sc));
    }
    uint8_t* cache = reinterpret_cast<uint8_t*>(is_k ? p.k_cache : p.v_cache);
    const uint2 codes = make_uint2((uint32_t)q[0] | ((uint32_t)q[1] << 16),
                                   (uint32_t)q[2] | ((uint32_t)q[3] << 16));
    *reinterpret_cast<uint2*>(cache + dst + 8 * c) = codes;
    return make_uint4(codes.x, codes.y, 0u, 0u);
}

// The wait limit of the pipeline barriers (a test build can shorten it).
#ifdef PA_TEST_HOOKS
#define PA_DECODE_WAIT_LIMIT(p) ((p).test_wait_limit_ns)
#else
#define PA_DECODE_WAIT_LIMIT(p) kWaitLimitNs
#endif

template <typename T, int D, int kMode, bool kFp8 = false>
__global__ void __launch_bounds__(kDecodeThreads, kFp8 ? kMinCtasPerSmFp8 : kMinCtasPerSm)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v,
                        const __grid_constant__ DecodeParams p) {
    using Lay = DecodeLayout<D, kFp8>;
    using M = Mma<T>;
    static_assert(!kFp8 || D == 128, "the FP8 cache is built for head_dim 128");
    constexpr int kKSteps = D / 16;     // 16-dim slices of D

    constexpr bool kPartitioned = kMode != kModeSingle;
    __shared__ __align__(8) uint64_t full_bar[Lay::kRing];
    __shared__ __align__(8) uint64_t empty_bar[Lay::kRing];
    __shared__ int merge_here;          // fused step: this CTA merges the partitions
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    // Grid (sequences, KV heads, partitions): sequences vary fastest, so CTAs
    // launch partition by partition -- every first partition, then every
    // second one, ...; the later, shorter last partitions of long sequences
    // come at the end, which keeps the tail of the grid short.
    const int b = blockIdx.x;
    const int g = blockIdx.y;
    const int part = blockIdx.z;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int G = p.group;

    grid_dependency_wait();          // inputs may come from the previous kernel
    allow_dependent_launch();

    // Context length, bounded so the table row is never overrun.
    const int max_ctx = p.max_blocks_per_seq * p.block_size;
    int L = p.context_lens[b];
    if (L < 0 || L > max_ctx) {
        if (threadIdx.x == 0 && part == 0 && g == 0) flag_error(p.err, PA_DEVERR_BAD_CONTEXT);
        L = L < 0 ? 0 : max_ctx;
    }
    int t_begin = 0, t_end = L, parts = 1;
    if (kPartitioned) {
        parts = min((L + p.partition_tokens - 1) / p.partition_tokens, p.max_parts);
        t_begin = part * p.partition_tokens;
        if (kMode == kModeStep && L == 0 && part == 0) {
            // Empty context: zero output; a new token cannot belong to it.
            T* out = reinterpret_cast<T*>(p.out) + ((size_t)b * p.num_q_heads + (size_t)g * G) * D;
            for (int i = threadIdx.x; i < G * D; i += blockDim.x) out[i] = from_float<T>(0.f);
            if (threadIdx.x == 0 && g == 0 && p.slot_mapping[b] >= 0)
                flag_error(p.err, PA_DEVERR_BAD_SLOT);
            return;
        }
        if (t_begin >= L) return;                       // partition past the end
        t_end = min(t_begin + p.partition_tokens, L);
    } else if (L == 0) {
        // Empty context: zero output for the group's heads.
        T* out = reinterpret_cast<T*>(p.out) + ((size_t)b * p.num_q_heads + (size_t)g * G) * D;
        for (int i = threadIdx.x; i < G * D; i += blockDim.x) out[i] = from_float<T>(0.f);
        return;
    }
    const int tile_begin = t_begin / kTileTokens;                  // t_begin % 16 == 0
    const int n_tiles = (t_end + kTileTokens - 1) / kTileTokens - tile_begin;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Lay::kRing; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------------
        // producer: block table -> TMA boxes
        // ------------------------------------------------------------------
        if (lane == 0) {
            prefetch_tensor_map(&tmap_k);
            prefetch_tensor_map(&tmap_v);
        }
        const int32_t* table = p.block_tables + (size_t)b * p.max_blocks_per_seq;
        const int tiles_per_block = p.block_size / kTileTokens;
        int issue_end = n_tiles;                        // tiles this producer issues
#ifdef PA_TEST_HOOKS
        if ((long long)blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y *
                                                            blockIdx.z) == p.test_cta)
            issue_end = min(n_tiles, max(0, p.test_tile));
#endif
        // Tiles go out in rounds of kBatch: in a round, lane t * kBoxes + j
        // issues box j (K halves, then V halves) of tile i + t after waiting
        // itself for that tile's stage, so one warp instruction issues every
        // box of the round.  With one issuing lane the stage wait, the byte
        // count and each copy are paid in sequence, ~600-750 cycles a tile,
        // which is what held a CTA streaming alone over an FP8 cache to
        // 12 GB/s (17 GB/s in rounds of two).  Lane l holds the table
        // entries of tiles i0 + l (blk) and i0 + 32 + l (blk_next, read a
        // chunk ahead so a new chunk does not wait for the table).
        constexpr int kBoxes = 2 * Lay::kHalves;
        constexpr int kBatch = kIssueBatch < Lay::kRing ? kIssueBatch : Lay::kRing;
        static_assert(kBatch * kBoxes <= 32 && 32 % kBatch == 0, "a round fits one warp");
        const int t_lane = lane / kBoxes, box = lane % kBoxes;
        const int hh = box % Lay::kHalves;
        const bool is_v = box >= Lay::kHalves;
        const CUtensorMap* tmap = is_v ? &tmap_v : &tmap_k;
        auto entry = [&](int tile) {
            int e = 0;
            if (tile < n_tiles) {
                e = __ldg(table + (tile_begin + tile) / tiles_per_block);
                if (e < 0 || e >= p.num_blocks) flag_error(p.err, PA_DEVERR_BAD_CONTEXT);
            }
            return e;
        };
        int blk = entry(lane);
        int blk_next = entry(32 + lane);
        bool ok = true;
        for (int i0 = 0; i0 < issue_end && ok; i0 += 32) {
            if (i0 > 0) {
                blk = blk_next;
                blk_next = entry(i0 + 32 + lane);
            }
            const int cnt = min(32, issue_end - i0);
            for (int k = 0; k < cnt; k += kBatch) {
                const int pblk = __shfl_sync(0xffffffffu, blk, (k + t_lane) & 31);
                const int it = i0 + k + t_lane;
                const bool act = t_lane < kBatch && k + t_lane < cnt;
                const int st = it % Lay::kRing;
                bool good = true;
                if (act && it >= Lay::kRing)
                    good = mbar_wait(&empty_bar[st], ((it / Lay::kRing) - 1) & 1,
                                     PA_DECODE_WAIT_LIMIT(p));
                if (act && good && box == 0) mbar_arrive_expect_tx(&full_bar[st], Lay::kStageBytes);
                // the vote also puts every expect_tx of the round before its copies
                if (!__all_sync(0xffffffffu, good)) {
                    if (lane == 0) flag_error(p.err, PA_DEVERR_WAIT_TIMEOUT);
                    ok = false;
                    break;
                }
                if (act) {
                    const int sub = ((tile_begin + it) % tiles_per_block) * kTileTokens;
                    uint8_t* dst = smem + st * Lay::kStageBytes + (is_v ? Lay::kTileBytes : 0) +
                                   hh * Lay::kBoxBytes;
                    tma_load_4d(dst, tmap, &full_bar[st], hh * kBoxElems, g, sub, pblk);
                }
            }
        }
        return;
    }

    // ----------------------------------------------------------------------
    // consumers
    // ----------------------------------------------------------------------
    // Fragment roles (m16n8k16, r = lane/4, c = lane%4):
    //   S^T[t][h] = K[t][:] . q[h][:]   A = K tile (16 tokens x 16 dims),
    //                                   B = q^T (16 dims x 8 heads)
    //   O^T[d][h] += V^T[d][:] . P^T[:][h]  A = V^T (16 dims x 16 tokens),
    //                                   B = P^T (16 tokens x 8 heads)
    // so each thread holds scores of tokens r and r+8 for heads 2c, 2c+1 and
    // accumulators of dims r, r+8 (per 16-dim slab) for the same two heads.
    const int r8 = lane >> 2;
    const int c4 = lane & 3;
    const int hA = 2 * c4, hB = 2 * c4 + 1;      // this thread's two heads

    uint32_t qb[kKSteps][2];
    float scale_log2 = p.scale_log2;
    {
        const T* qg = reinterpret_cast<const T*>(p.q) + ((size_t)b * p.num_q_heads + (size_t)g * G) * D;
        if constexpr (kFp8) {
            const int sq = load_q_fragments_fp8<T>(qb, qg, G, lane);   // q / 2^sq in fp16
            scale_log2 *= __int_as_float((127 + sq) << 23);
        } else {
            load_q_fragments<T, D>(qb, qg, G, lane);
        }
    }
    // The fragments go to shared memory (both consumer warps hold the same
    // ones) and are read back per k-step: the 16 registers they would pin
    // through the tile loop are what made the fused step spill.
    const uint32_t q_lane = smem_u32(smem + Lay::kBodyBytes) + lane * 8;
    if (warp == 0) {
#pragma unroll
        for (int kk = 0; kk < kKSteps; ++kk)
            asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(q_lane + kk * 256), "r"(qb[kk][0]),
                         "r"(qb[kk][1])
                         : "memory");
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    auto qfrag = [&](int kk, uint32_t& b0, uint32_t& b1) { lds64(q_lane + kk * 256, b0, b1); };
    TileState<D> ts;
    ts.reset();

    // Fused step: the CTA of the last partition owns the sequence's new token
    // (position L - 1).  It checks that slot_mapping[b] is that position's
    // slot, writes the token's K/V for this KV head into the cache, and puts
    // them into the staged tile in place of what the TMA read there.
    int64_t new_slot = -1;
    int new_tile = -1;                      // CTA-local tile index, -1: not attended here
    if (kMode == kModeStep && part == parts - 1) {
        const int64_t slot = p.slot_mapping[b];
        if (slot >= 0) {
            const int pos = L - 1;
            const int64_t blk = p.block_tables[(size_t)b * p.max_blocks_per_seq + pos / p.block_size];
            const int64_t want = blk * p.block_size + pos % p.block_size;
            if (slot == want && blk >= 0 && blk < p.num_blocks) {
                new_slot = slot;
                if (pos < t_end) new_tile = pos / kTileTokens - tile_begin;
            } else if (warp == 0 && lane == 0) {
                flag_error(p.err, PA_DEVERR_BAD_SLOT);
            }
        }
    }

    if constexpr (kFp8) {
        // Consumer warp w takes the tile pairs (2i, 2i + 1), i = w, w + W, ...
        // (W consumer warps); tile t sits in stage t % kRing, so with kRing a
        // multiple of 2W every stage belongs to exactly one warp.
        static_assert(Lay::kRing % (2 * kConsumerWarps) == 0, "FP8 stages must pair up per warp");
        for (int it = 2 * warp; it < n_tiles; it += 2 * kConsumerWarps) {
            const bool two = it + 1 < n_tiles;
            const int st0 = it % Lay::kRing, st1 = (it + 1) % Lay::kRing;
            bool ok = mbar_wait(&full_bar[st0], (it / Lay::kRing) & 1, PA_DECODE_WAIT_LIMIT(p));
            if (ok && two)
                ok = mbar_wait(&full_bar[st1], ((it + 1) / Lay::kRing) & 1, PA_DECODE_WAIT_LIMIT(p));
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) flag_error(p.err, PA_DEVERR_WAIT_TIMEOUT);
                break;
            }
            uint8_t* ktile0 = smem + st0 * Lay::kStageBytes;
            uint8_t* vtile0 = ktile0 + Lay::kTileBytes;
            uint8_t* ktile1 = smem + st1 * Lay::kStageBytes;
            uint8_t* vtile1 = ktile1 + Lay::kTileBytes;
            if (kMode == kModeStep && (it == new_tile || (two && it + 1 == new_tile))) {
                // lanes 0-15: 8-code chunks of K, lanes 16-31: of V, into the staged codes
                const int c = lane & 15;
                const bool is_k = lane < 16;
                const bool first = it == new_tile;
                const uint4 cv = new_token_chunk<T, D, true>(p, b, g, new_slot, c, is_k);
                put_code_chunk(is_k ? (first ? ktile0 : ktile1) : (first ? vtile0 : vtile1),
                               (L - 1) % kTileTokens, c, make_uint2(cv.x, cv.y));
                fence_proxy_async_smem();
                __syncwarp();
            }
            const int tok0 = (tile_begin + it) * kTileTokens;
            if (two) {
                attend_pair_fp8(ts, qfrag, ktile0, vtile0, ktile1, vtile1, tok0, t_end, scale_log2,
                                lane, [&] {
                                    fence_proxy_async_smem();
                                    __syncwarp();
                                    if (lane == 0) {
                                        mbar_arrive(&empty_bar[st0]);
                                        mbar_arrive(&empty_bar[st1]);
                                    }
                                });
            } else {
                attend_tile_fp8(ts, qfrag, ktile0, vtile0, tok0, t_end, scale_log2, lane,
                                [&] { release_stage(&empty_bar[st0], lane); });
            }
        }
    } else {
        for (int it = warp; it < n_tiles; it += kConsumerWarps) {
            const int st = it % Lay::kRing;
            bool ok = mbar_wait(&full_bar[st], (it / Lay::kRing) & 1, PA_DECODE_WAIT_LIMIT(p));
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) flag_error(p.err, PA_DEVERR_WAIT_TIMEOUT);
                break;
            }
            uint8_t* ktile = smem + st * Lay::kStageBytes;
            uint8_t* vtile = ktile + Lay::kTileBytes;
            if (kMode == kModeStep && it == new_tile) {
                // lanes 0-15: 16-byte chunks of K, lanes 16-31: of V
                const int c = lane & 15;
                if (c < D / 8) {
                    const bool is_k = lane < 16;
                    put_tile_chunk(is_k ? ktile : vtile, (L - 1) % kTileTokens, c,
                                   new_token_chunk<T, D, false>(p, b, g, new_slot, c, is_k));
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            attend_tile<T, D>(ts, qfrag, ktile, vtile, (tile_begin + it) * kTileTokens, t_end,
                              scale_log2, lane);
            release_stage(&empty_bar[st], lane);
        }
    }

    if (kMode == kModeStep && new_slot >= 0 && new_tile < 0 && warp == 0) {
        const int c = lane & 15;
        if (c < D / 8) (void)new_token_chunk<T, D, kFp8>(p, b, g, new_slot, c, lane < 16);
    }

    ts.reduce_row_sums();

    // ----------------------------------------------------------------------
    // merge the consumer warps
    // ----------------------------------------------------------------------
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");   // pipeline drained
    float* mrg = reinterpret_cast<float*>(smem);
    {
        float* wo = mrg + warp * Lay::kMergeFloatsPerWarp;
#pragma unroll
        for (int n = 0; n < kKSteps; ++n) {
            int d_lo = 16 * n + r8, d_hi = d_lo + 8;        // rows r8, r8 + 8 of slab n
            if constexpr (kFp8) fp8_dims(n, r8, d_lo, d_hi);
            if (hA < G) {
                wo[hA * D + d_lo] = ts.acc[n][0];
                wo[hA * D + d_hi] = ts.acc[n][2];
            }
            if (hB < G) {
                wo[hB * D + d_lo] = ts.acc[n][1];
                wo[hB * D + d_hi] = ts.acc[n][3];
            }
        }
        if (r8 == 0) {
            if (hA < G) {
                wo[kMaxGroup * D + hA] = ts.mA;
                wo[kMaxGroup * D + kMaxGroup + hA] = ts.lA;
                wo[kMaxGroup * D + 2 * kMaxGroup + hA] = ts.tA;
            }
            if (hB < G) {
                wo[kMaxGroup * D + hB] = ts.mB;
                wo[kMaxGroup * D + kMaxGroup + hB] = ts.lB;
                wo[kMaxGroup * D + 2 * kMaxGroup + hB] = ts.tB;
            }
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");

    const int tid = threadIdx.x;                      // 0..127
    const int items = G * (D / 4);                    // 4 output dims per item
    for (int item = tid; item < items; item += kConsumerWarps * 32) {
        const int h = item / (D / 4);
        const int d = (item - h * (D / 4)) * 4;
        float mref = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w)
            mref = fmaxf(mref, mrg[w * Lay::kMergeFloatsPerWarp + kMaxGroup * D + h]);
        float den = 0.f, o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f, mt = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float* wo = mrg + w * Lay::kMergeFloatsPerWarp;
            const float mw = wo[kMaxGroup * D + h];
            const float f = (mw == -INFINITY) ? 0.f : ex2(mw - mref);
            den += f * wo[kMaxGroup * D + kMaxGroup + h];
            const float4 v = *reinterpret_cast<const float4*>(wo + h * D + d);
            o0 += f * v.x;
            o1 += f * v.y;
            o2 += f * v.z;
            o3 += f * v.w;
            mt = fmaxf(mt, wo[kMaxGroup * D + 2 * kMaxGroup + h]);
        }
        const float inv = (kFp8 ? p.v_scale : 1.f) / den;
        const size_t qh = (size_t)b * p.num_q_heads + (size_t)g * G + h;
        if (kMode == kModeSplit || (kMode == kModeStep && parts > 1)) {
            const size_t idx = qh * p.max_parts + part;
            *reinterpret_cast<float4*>(p.tmp_out + idx * D + d) =
                make_float4(o0 * inv, o1 * inv, o2 * inv, o3 * inv);
            if (d == 0) {
                p.max_logits[idx] = mt * kLn2;
                p.exp_sums[idx] = den * ex2(mref - mt);
            }
        } else {
            T* out = reinterpret_cast<T*>(p.out) + qh * D + d;
            const uint32_t lo = M::pack(o0 * inv, o1 * inv);
            const uint32_t hi = M::pack(o2 * inv, o3 * inv);
            *reinterpret_cast<uint2*>(out) = make_uint2(lo, hi);
        }
    }

    if (kMode == kModeStep && parts > 1) {
        // The last CTA of the (sequence, KV head) to finish merges all
        // partitions: M = max m_s, w_s = l_s e^(m_s - M), out = sum w_s o_s / sum w_s.
        // Its chain is on the launch's critical path (the longest partition
        // of a sequence finishes last), so it is kept to two round trips:
        // the count, then every partition's record loaded at once.
        // Release / acquire: the barrier orders this CTA's partial-record
        // writes before thread 0's acq_rel add, and the add that sees
        // parts - 1 acquires every other partition's records for the threads
        // that pass the next barrier.
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
        int* counter = p.counters + (size_t)b * p.num_kv_heads + g;
        if (tid == 0) {
            int before;
            asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                         : "=r"(before)
                         : "l"(counter)
                         : "memory");
            merge_here = before == parts - 1;
        }
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
        if (!merge_here) return;
        const size_t qh0 = (size_t)b * p.num_q_heads + (size_t)g * G;
        for (int item = tid; item < items; item += kConsumerWarps * 32) {
            const int h = item / (D / 4);
            const int d = (item - h * (D / 4)) * 4;
            const float* ml = p.max_logits + (qh0 + h) * p.max_parts;
            const float* es = p.exp_sums + (qh0 + h) * p.max_parts;
            const float* src = p.tmp_out + (qh0 + h) * p.max_parts * D + d;
            // partitions four at a time, each group's loads issued together,
            // folded in with a running maximum (natural-log units)
            float mx = -INFINITY, den = 0.f;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int s0 = 0; s0 < parts; s0 += 4) {
                float mj[4], ej[4];
                float4 xj[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const bool in = s0 + j < parts;
                    mj[j] = in ? __ldcg(ml + s0 + j) : -INFINITY;
                    ej[j] = in ? __ldcg(es + s0 + j) : 0.f;
                    xj[j] = in ? __ldcg(reinterpret_cast<const float4*>(src + (size_t)(s0 + j) * D))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                const float nm = fmaxf(fmaxf(mx, fmaxf(mj[0], mj[1])), fmaxf(mj[2], mj[3]));
                const float keep = __expf(mx - nm);               // 0 on the first group
                den *= keep;
                acc.x *= keep; acc.y *= keep; acc.z *= keep; acc.w *= keep;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float wj = ej[j] * __expf(mj[j] - nm);  // 0 past the last partition
                    den += wj;
                    acc.x += wj * xj[j].x; acc.y += wj * xj[j].y;
                    acc.z += wj * xj[j].z; acc.w += wj * xj[j].w;
                }
                mx = nm;
            }
            const float inv = 1.f / den;
            T* out = reinterpret_cast<T*>(p.out) + (qh0 + h) * D + d;
            const uint32_t lo = M::pack(acc.x * inv, acc.y * inv);
            const uint32_t hi = M::pack(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2*>(out) = make_uint2(lo, hi);
        }
        if (tid == 0) *counter = 0;                        // ready for the next step
    }
}

template <typename T, int D, int kMode, bool kFp8 = false>
cudaError_t launch_decode_mode(const CUtensorMap& tmk, const CUtensorMap& tmv,
                               const DecodeParams& p, dim3 grid, cudaStream_t stream) {
    const int smem = DecodeLayout<D, kFp8>::kDynamicSmem;
    cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel<T, D, kMode, kFp8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = launch_with_pdl(paged_decode_kernel<T, D, kMode, kFp8>, grid, dim3(kDecodeThreads), smem,
                        stream, tmk, tmv, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t launch_decode_t(int mode, const CUtensorMap& tmk, const CUtensorMap& tmv,
                            const DecodeParams& p, dim3 grid, cudaStream_t stream) {
    if (mode == kModeSplit) return launch_decode_mode<T, D, kModeSplit>(tmk, tmv, p, grid, stream);
    if (mode == kModeStep) return launch_decode_mode<T, D, kModeStep>(tmk, tmv, p, grid, stream);
    return launch_decode_mode<T, D, kModeSingle>(tmk, tmv, p, grid, stream);
}

template <typename T>
cudaError_t launch_decode_fp8_t(int mode, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                const DecodeParams& p, dim3 grid, cudaStream_t stream) {
    if (mode == kModeSplit)
        return launch_decode_mode<T, 128, kModeSplit, true>(tmk, tmv, p, grid, stream);
    if (mode == kModeStep)
        return launch_decode_mode<T, 128, kModeStep, true>(tmk, tmv, p, grid, stream);
    return launch_decode_mode<T, 128, kModeSingle, true>(tmk, tmv, p, grid, stream);
}

}  // namespace pa
