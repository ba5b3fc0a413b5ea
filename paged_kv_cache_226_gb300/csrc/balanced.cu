// Work-balanced fused decode layer-step.
//
// The partitioned kernels give every (sequence, KV head, partition) its own
// CTA; for batches of many short contexts that means more than one wave of
// CTAs, and the CTAs that start last stream their partition alone at the end
// of the launch, each limited by the few tiles it can keep in flight.  Here
// the work is balanced instead: the tiles of all (sequence, KV head)
// segments, in order, form one sequence of N 16-token tiles, and warp w of a
// single wave of CTAs streams tiles [w*Q, (w+1)*Q) with Q = ceil(N / warps),
// so every warp runs from the start of the launch to its end.  Each warp
// issues the TMA loads of its own range into a private ring (no producer
// warp, no cross-warp coupling: a warp that stops to merge holds up only its
// own stream, whose next tiles are already in flight).  A warp crosses
// segment boundaries without draining its ring; each segment piece it covers
// yields a partial result, and the last warp to finish a segment merges the
// pieces (log-sum-exp) into the output.  A one-CTA plan kernel first scans
// the per-sequence tile counts.
//
// The cache write of the new token and its use by attention follow the
// fused step (pa_decode_step).
#include "decode_tile.cuh"

namespace pa {

constexpr int kPlanThreads = 1024;

// plan[0] = N (total tiles), plan[1] = Q (tiles per warp), plan[2 + b] =
// exclusive prefix of T_b = ceil(L_b / 16) over sequences (B + 1 entries).
// Sequences with L_b = 0 get a zero output here (no tiles reach them).
template <typename T, int D>
__global__ void __launch_bounds__(kPlanThreads)
    balanced_plan_kernel(const __grid_constant__ BalancedParams p) {
    grid_dependency_wait();
    allow_dependent_launch();
    __shared__ int warp_sums[kPlanThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int B = p.num_seqs;
    const int max_ctx = p.max_blocks_per_seq * p.block_size;
    const int per = (B + kPlanThreads - 1) / kPlanThreads;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
    int local = 0;
    for (int b = b0; b < b1; ++b) {
        int L = p.context_lens[b];
        if (L < 0 || L > max_ctx) {
            flag_error(p.err, PA_DEVERR_BAD_CONTEXT);
            L = L < 0 ? 0 : max_ctx;
        }
        local += (L + kTileTokens - 1) / kTileTokens;
        if (L == 0) {
            T* out = reinterpret_cast<T*>(p.out) + (size_t)b * p.num_q_heads * D;
            for (int i = 0; i < p.num_q_heads * D; ++i) out[i] = from_float<T>(0.f);
            if (p.slot_mapping[b] >= 0) flag_error(p.err, PA_DEVERR_BAD_SLOT);
        }
    }
    // block-wide exclusive scan of the per-thread sums
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sums[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int v = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += y;
        }
        warp_sums[lane] = v;                         // inclusive over warps
    }
    __syncthreads();
    int run = incl - local + (wid > 0 ? warp_sums[wid - 1] : 0);
    int* prefix = p.plan + 2;
    for (int b = b0; b < b1; ++b) {
        prefix[b] = run;
        int L = p.context_lens[b];
        L = L < 0 ? 0 : (L > max_ctx ? max_ctx : L);
        run += (L + kTileTokens - 1) / kTileTokens;
    }
    const long long total = (long long)warp_sums[kPlanThreads / 32 - 1];
    const long long N = total * p.num_kv_heads;
    const int Q = (int)max(1LL, (N + p.num_warps - 1) / p.num_warps);
    if (tid == kPlanThreads - 1) {
        prefix[B] = (int)total;
        p.plan[0] = (int)N;
        p.plan[1] = Q;
    }
    __syncthreads();                                 // prefix[] written by this CTA
    // start cursor (b, g, t, T) of every warp slot's range
    int4* starts = reinterpret_cast<int4*>(p.plan + plan_starts_offset(B));
    for (int ws = tid; ws < p.num_warps; ws += kPlanThreads) {
        const long long x = (long long)ws * Q;
        if (x >= N) continue;
        const long long key = x / p.num_kv_heads;
        int lo = 0, hi = B;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if ((long long)prefix[mid] > key) hi = mid; else lo = mid + 1;
        }
        const int b = lo - 1;
        const int Tb = prefix[b + 1] - prefix[b];
        const long long off = x - (long long)p.num_kv_heads * prefix[b];
        const int g = (int)(off / Tb);
        starts[ws] = make_int4(b, g, (int)(off - (long long)g * Tb), Tb);
    }
}

// Position of a tile in the (sequence, KV head, tile) order.
struct TileCursor {
    int b, g, t, T;           // sequence, KV head, tile within the segment, tiles of b

    // Moves n >= 0 tiles forward (stops at the end of the batch).
    __device__ __forceinline__ void advance(int n, const int* prefix, int B, int Hkv) {
        while (n > 0) {
            const int left = T - t;
            if (n < left) {
                t += n;
                return;
            }
            n -= left;
            t = 0;
            if (++g == Hkv) {
                g = 0;
                do {
                    if (++b >= B) return;
                    T = __ldg(prefix + b + 1) - __ldg(prefix + b);
                } while (T == 0);
            }
        }
    }

    __device__ __forceinline__ void load(const int* plan, int B, long long ws) {
        const int4 v = __ldcg(reinterpret_cast<const int4*>(plan + plan_starts_offset(B)) + ws);
        b = v.x, g = v.y, t = v.z, T = v.w;
    }

    __device__ __forceinline__ long long seg_start(const int* prefix, int Hkv) const {
        return (long long)Hkv * __ldg(prefix + b) + (long long)g * T;
    }
};

template <int D, bool kFp8>
struct StreamLayout {
    static constexpr int kHalves = kFp8 ? 1 : D / kBoxElems;
    static constexpr int kTileBytes = kHalves * kBox16Bytes;       // K or V of one tile
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kTile16Bytes = (D / kBoxElems) * kBox16Bytes;
    static constexpr int kConvBytes = 0;     // FP8 codes go from the stage to registers
    static constexpr int kRing = (kStreamRingBytes - kConvBytes) / kStageBytes;  // stages
    static constexpr int kWarpBytes = kRing * kStageBytes + kConvBytes;
    static constexpr int kDynamicSmem = kStreamWarps * kWarpBytes + 1024;
    static_assert(kRing >= 2, "a warp needs at least two stages");
    static_assert(kWarpBytes % 1024 == 0, "warp rings must keep the 128-byte swizzle alignment");
};

// Writes the fused step's new token (chunk c of K or V, head g) into the
// cache and returns it as staged data: the 16-bit values, or for an FP8
// cache its eight E4M3 codes in .x and .y.
template <typename T, int D, bool kFp8>
__device__ __forceinline__ uint4 balanced_new_token(const BalancedParams& p, int b, int g,
                                                    int64_t slot, int c, bool is_k) {
    const size_t row = ((size_t)b * p.num_kv_heads + g) * D;
    const uint4 val = __ldg(reinterpret_cast<const uint4*>(
                                reinterpret_cast<const T*>(is_k ? p.k_new : p.v_new) + row) + c);
    const size_t dst = ((size_t)slot * p.num_kv_heads + g) * D;
    if (!kFp8) {
        reinterpret_cast<uint4*>(reinterpret_cast<T*>(is_k ? p.k_cache : p.v_cache) + dst)[c] = val;
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

// Log-sum-exp merge of the np pieces (records wfirst + j + z) of segment z by
// one warp.  Lanes take pieces for the per-head maxima and weights; for the
// weighted sum each lane owns D/32 dims of every head and keeps two pieces'
// worth of loads (all heads) in flight.
template <int V>
__device__ __forceinline__ void load_vec(float (&x)[V], const float* src) {
    if constexpr (V == 4) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(src));
        x[0] = v.x, x[1] = v.y, x[2] = v.z, x[3] = v.w;
    } else {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(src));
        x[0] = v.x, x[1] = v.y;
    }
}

template <typename T, int D>
__device__ __forceinline__ void merge_pieces(const BalancedParams& p, int z, long long wfirst,
                                             int np, size_t qh0, int G, int lane) {
    constexpr int V = D / 32;
    float mx[kMaxGroup], den[kMaxGroup], acc[kMaxGroup][V];
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
        mx[h] = -INFINITY;
        den[h] = 0.f;
#pragma unroll
        for (int e = 0; e < V; ++e) acc[h][e] = 0.f;
    }
    for (int j = lane; j < np; j += 32) {
        const size_t r = (size_t)(wfirst + j + z) * G;
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h)
            if (h < G) mx[h] = fmaxf(mx[h], __ldcg(p.rec_m + r + h));
    }
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], o));
    }
    for (int j0 = 0; j0 < np; j0 += 32) {
        const int j = j0 + lane;
        float w[kMaxGroup];
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h) w[h] = 0.f;
        if (j < np) {
            const size_t r = (size_t)(wfirst + j + z) * G;
#pragma unroll
            for (int h = 0; h < kMaxGroup; ++h)
                if (h < G) w[h] = __ldcg(p.rec_l + r + h) * ex2(__ldcg(p.rec_m + r + h) - mx[h]);
        }
#pragma unroll
        for (int h = 0; h < kMaxGroup; ++h) den[h] += w[h];
        const int n = min(32, np - j0);
        for (int i = 0; i < n; i += 2) {
            float x[2][kMaxGroup][V];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const size_t r = (size_t)(wfirst + j0 + min(i + u, n - 1) + z) * G;
                const float* src = p.rec_o + r * D + lane * V;
#pragma unroll
                for (int h = 0; h < kMaxGroup; ++h)
                    if (h < G) load_vec<V>(x[u][h], src + h * D);
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                if (i + u < n) {
#pragma unroll
                    for (int h = 0; h < kMaxGroup; ++h) {
                        if (h < G) {
                            const float wt = __shfl_sync(0xffffffffu, w[h], i + u);
#pragma unroll
                            for (int e = 0; e < V; ++e) acc[h][e] += wt * x[u][h][e];
                        }
                    }
                }
            }
        }
    }
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
        if (h < G) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) den[h] += __shfl_xor_sync(0xffffffffu, den[h], o);
            T* out = reinterpret_cast<T*>(p.out) + (qh0 + h) * D + lane * V;
#pragma unroll
            for (int e = 0; e < V; ++e) out[e] = from_float<T>(acc[h][e] / den[h]);
        }
    }
}

template <typename T, int D, bool kFp8>
__global__ void __launch_bounds__(kStreamWarps * 32, kStreamCtasPerSm)
    balanced_step_kernel(const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v,
                         const __grid_constant__ BalancedParams p) {
    using Lay = StreamLayout<D, kFp8>;
    constexpr int R = Lay::kRing;
    static_assert(!kFp8 || D == 128, "the FP8 cache is built for head_dim 128");
    __shared__ __align__(8) uint64_t full_bar[kStreamWarps][R];
    __shared__ int stage_blk[kStreamWarps][R];          // physical block of each staged tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ring = smem + warp * Lay::kWarpBytes;
    uint64_t* full = full_bar[warp];
    int* sblk = stage_blk[warp];

    // the warp's own barriers and the tensor maps, before the inputs are ready
    if (lane == 0) {
        for (int s = 0; s < R; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
        if (warp == 0) {
            prefetch_tensor_map(&tmap_k);
            prefetch_tensor_map(&tmap_v);
        }
    }
    __syncwarp();
    grid_dependency_wait();                  // the plan and the inputs are ready
    allow_dependent_launch();

    const int B = p.num_seqs, Hkv = p.num_kv_heads, G = p.group;
    const int* prefix = p.plan + 2;
    const long long N = p.plan[0];
    const int Q = p.plan[1];
    const long long ws = (long long)blockIdx.x * kStreamWarps + warp;
    const long long x0 = ws * Q;
    const int count = (int)max(0LL, min((long long)Q, N - x0));
    if (count == 0) return;
    const int max_ctx = p.max_blocks_per_seq * p.block_size;
    const int tiles_per_block = p.block_size / kTileTokens;
    const int r8 = lane >> 2, c4 = lane & 3;
    const int hA = 2 * c4, hB = 2 * c4 + 1;

    TileCursor cur;                          // the tile being attended
    cur.load(p.plan, B, ws);

    // ------------------------------------------------------------------
    // load side: descriptors (block, KV head, token offset) of 32 tiles at a
    // time, one per lane: set A holds the batch being issued, set B the next
    // one, whose table reads have 32 issues' time to land.
    // ------------------------------------------------------------------
    TileCursor bc = cur;                     // first tile of the next batch to describe
    int a_blk = 0, a_g = 0, a_sub = 0, b_blk = 0, b_g = 0, b_sub = 0;
    auto describe = [&](int i0, int& blk, int& gg, int& sub) {
        blk = 0, gg = 0, sub = 0;
        if (i0 >= count) return;
        TileCursor c = bc;
        c.advance(lane, prefix, B, Hkv);
        if (i0 + lane < count) {
            blk = __ldg(p.block_tables + (size_t)c.b * p.max_blocks_per_seq + c.t / tiles_per_block);
            gg = c.g;
            sub = (c.t % tiles_per_block) * kTileTokens;
        }
        c.advance(1, prefix, B, Hkv);
        bc.b = __shfl_sync(0xffffffffu, c.b, 31);
        bc.g = __shfl_sync(0xffffffffu, c.g, 31);
        bc.t = __shfl_sync(0xffffffffu, c.t, 31);
        bc.T = __shfl_sync(0xffffffffu, c.T, 31);
    };
    describe(0, a_blk, a_g, a_sub);
    describe(32, b_blk, b_g, b_sub);
    // Tile j of the range into stage j % R (whole warp; lane 0 issues).
    auto issue = [&](int j) {
        if (j > 0 && (j & 31) == 0) {
            a_blk = b_blk, a_g = b_g, a_sub = b_sub;
            describe(j + 32, b_blk, b_g, b_sub);
        }
        const int blk = __shfl_sync(0xffffffffu, a_blk, j & 31);
        const int gg = __shfl_sync(0xffffffffu, a_g, j & 31);
        const int sub = __shfl_sync(0xffffffffu, a_sub, j & 31);
        if (lane == 0) {
            if (blk < 0 || blk >= p.num_blocks) flag_error(p.err, PA_DEVERR_BAD_CONTEXT);
            const int st = j % R;
            sblk[st] = blk;
            uint8_t* kdst = ring + st * Lay::kStageBytes;
            uint8_t* vdst = kdst + Lay::kTileBytes;
            mbar_arrive_expect_tx(&full[st], Lay::kStageBytes);
#pragma unroll
            for (int hh = 0; hh < Lay::kHalves; ++hh) {
                tma_load_4d(kdst + hh * kBox16Bytes, &tmap_k, &full[st], hh * kBoxElems, gg, sub,
                            blk);
                tma_load_4d(vdst + hh * kBox16Bytes, &tmap_v, &full[st], hh * kBoxElems, gg, sub,
                            blk);
            }
        }
    };
    for (int j = 0; j < R && j < count; ++j) issue(j);

    // ------------------------------------------------------------------
    // attention over the range, piece by piece
    // ------------------------------------------------------------------
    const T* qbase = reinterpret_cast<const T*>(p.q);
    uint32_t qb[D / 16][2], qn[D / 16][2];
    TileState<D> ts;
    // the first piece's query rows, length and new-token slot; later pieces'
    // are prefetched during the last tile of the piece before
    // (FP8: fp16 fragments of q / 2^s in the FP8 dim order, s kept beside them)
    auto load_q = [&](uint32_t (&dst)[D / 16][2], const T* src) -> int {
        if constexpr (kFp8) {
            return load_q_fragments_fp8<T>(dst, src, G, lane);
        } else {
            load_q_fragments<T, D>(dst, src, G, lane);
            return 0;
        }
    };
    int sq_next = load_q(qn, qbase + ((size_t)cur.b * p.num_q_heads + (size_t)cur.g * G) * D);
    float scale_log2 = p.scale_log2;
    int L_next = p.context_lens[cur.b];
    int64_t slot_next = p.slot_mapping[cur.b];
    int L = 0;
    int64_t slot = -1;
    for (int k = 0; k < count; ++k) {
        const int b = cur.b, g = cur.g, t = cur.t;
        if (k == 0 || t == 0) {                          // a piece begins
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) qb[kk][0] = qn[kk][0], qb[kk][1] = qn[kk][1];
            scale_log2 = p.scale_log2 * __int_as_float((127 + sq_next) << 23);
            L = L_next < 0 ? 0 : (L_next > max_ctx ? max_ctx : L_next);
            slot = slot_next;
            ts.reset();
        }
        const bool piece_end = (k == count - 1) || (t == cur.T - 1);
        if (piece_end && k + 1 < count) {
            TileCursor nx = cur;
            nx.advance(1, prefix, B, Hkv);
            sq_next = load_q(qn, qbase + ((size_t)nx.b * p.num_q_heads + (size_t)nx.g * G) * D);
            L_next = p.context_lens[nx.b];
            slot_next = p.slot_mapping[nx.b];
        }
        const int st = k % R;
        bool ok = mbar_wait(&full[st], (k / R) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) flag_error(p.err, PA_DEVERR_WAIT_TIMEOUT);
            return;
        }
        const int blk = sblk[st];
        uint8_t* ktile = ring + st * Lay::kStageBytes;
        uint8_t* vtile = ktile + Lay::kTileBytes;
        if (slot >= 0 && t == (L - 1) / kTileTokens) {
            // the segment's last tile holds its new token (position L - 1)
            const int pos = L - 1;
            if (slot == (int64_t)blk * p.block_size + pos % p.block_size && blk >= 0 &&
                blk < p.num_blocks) {
                const int c = lane & 15;
                const bool is_k = lane < 16;
                if constexpr (kFp8) {
                    const uint4 cv = balanced_new_token<T, D, true>(p, b, g, slot, c, is_k);
                    put_code_chunk(is_k ? ktile : vtile, pos % kTileTokens, c,
                                   make_uint2(cv.x, cv.y));
                } else if (c < D / 8) {
                    put_tile_chunk(is_k ? ktile : vtile, pos % kTileTokens, c,
                                   balanced_new_token<T, D, false>(p, b, g, slot, c, is_k));
                }
                fence_proxy_async_smem();    // before a later TMA write of the stage
                __syncwarp();
            } else if (lane == 0 && g == 0) {
                flag_error(p.err, PA_DEVERR_BAD_SLOT);
            }
        }
        if constexpr (kFp8) {
            attend_tile_fp8(ts, qb, ktile, vtile, t * kTileTokens, L, scale_log2, lane, [&] {
                __syncwarp();                // the codes are in registers: refill the stage
                if (k + R < count) issue(k + R);
            });
        } else {
            attend_tile<T, D>(ts, qb, ktile, vtile, t * kTileTokens, L, scale_log2, lane);
            __syncwarp();
            if (k + R < count) issue(k + R);
        }

        if (piece_end) {
            ts.reduce_row_sums();
            const int z = b * Hkv + g;
            const long long s0 = cur.seg_start(prefix, Hkv);
            const long long wfirst = s0 / Q, wlast = (s0 + cur.T - 1) / Q;
            const size_t qh0 = (size_t)b * p.num_q_heads + (size_t)g * G;
            const float vsc = kFp8 ? p.v_scale : 1.f;
            const float iA = vsc / ts.lA, iB = vsc / ts.lB;
            if (wfirst == wlast) {
                // the whole segment: final output straight from the registers
                T* out = reinterpret_cast<T*>(p.out) + qh0 * D;
#pragma unroll
                for (int n = 0; n < D / 16; ++n) {
                    int d_lo = 16 * n + r8, d_hi = d_lo + 8;
                    if constexpr (kFp8) fp8_dims(n, r8, d_lo, d_hi);
                    if (hA < G) {
                        out[hA * D + d_lo] = from_float<T>(ts.acc[n][0] * iA);
                        out[hA * D + d_hi] = from_float<T>(ts.acc[n][2] * iA);
                    }
                    if (hB < G) {
                        out[hB * D + d_lo] = from_float<T>(ts.acc[n][1] * iB);
                        out[hB * D + d_hi] = from_float<T>(ts.acc[n][3] * iB);
                    }
                }
            } else {
                // partial record: normalised o, true max, sum at the true max (log2 units)
                const size_t rec = (size_t)(ws + z);
                float* ro = p.rec_o + rec * G * D;
#pragma unroll
                for (int n = 0; n < D / 16; ++n) {
                    int d_lo = 16 * n + r8, d_hi = d_lo + 8;
                    if constexpr (kFp8) fp8_dims(n, r8, d_lo, d_hi);
                    if (hA < G) {
                        ro[hA * D + d_lo] = ts.acc[n][0] * iA;
                        ro[hA * D + d_hi] = ts.acc[n][2] * iA;
                    }
                    if (hB < G) {
                        ro[hB * D + d_lo] = ts.acc[n][1] * iB;
                        ro[hB * D + d_hi] = ts.acc[n][3] * iB;
                    }
                }
                if (r8 == 0) {
                    if (hA < G) {
                        p.rec_m[rec * G + hA] = ts.tA;
                        p.rec_l[rec * G + hA] = ts.lA * ex2(ts.mA - ts.tA);
                    }
                    if (hB < G) {
                        p.rec_m[rec * G + hB] = ts.tB;
                        p.rec_l[rec * G + hB] = ts.lB * ex2(ts.mB - ts.tB);
                    }
                }
                __threadfence();
                __syncwarp();
                int last = 0;
                if (lane == 0) last = atomicAdd(p.counters + z, 1) == (int)(wlast - wfirst);
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
                    merge_pieces<T, D>(p, z, wfirst, (int)(wlast - wfirst + 1), qh0, G, lane);
                    if (lane == 0) p.counters[z] = 0;
                }
            }
        }
        cur.advance(1, prefix, B, Hkv);
    }
}

template <typename T, int D, bool kFp8>
cudaError_t launch_balanced_t(const CUtensorMap& tmk, const CUtensorMap& tmv,
                              const BalancedParams& p, int num_ctas, cudaStream_t stream) {
    cudaError_t e = launch_with_pdl(balanced_plan_kernel<T, D>, dim3(1), dim3(kPlanThreads), 0,
                                    stream, p);
    if (e != cudaSuccess) return e;
    const int smem = StreamLayout<D, kFp8>::kDynamicSmem;
    e = cudaFuncSetAttribute(balanced_step_kernel<T, D, kFp8>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_with_pdl(balanced_step_kernel<T, D, kFp8>, dim3(num_ctas),
                           dim3(kStreamWarps * 32), smem, stream, tmk, tmv, p);
}

cudaError_t launch_balanced(int dtype, int head_dim, bool fp8, const CUtensorMap& tmk,
                            const CUtensorMap& tmv, const BalancedParams& p, int num_ctas,
                            cudaStream_t stream) {
    if (fp8) {
        if (dtype == PA_BF16)
            return launch_balanced_t<__nv_bfloat16, 128, true>(tmk, tmv, p, num_ctas, stream);
        return launch_balanced_t<__half, 128, true>(tmk, tmv, p, num_ctas, stream);
    }
    if (dtype == PA_BF16) {
        if (head_dim == 64)
            return launch_balanced_t<__nv_bfloat16, 64, false>(tmk, tmv, p, num_ctas, stream);
        return launch_balanced_t<__nv_bfloat16, 128, false>(tmk, tmv, p, num_ctas, stream);
    }
    if (head_dim == 64) return launch_balanced_t<__half, 64, false>(tmk, tmv, p, num_ctas, stream);
    return launch_balanced_t<__half, 128, false>(tmk, tmv, p, num_ctas, stream);
}

}  // namespace pa
