// Work-balanced fused decode layer-step.
//
// The partitioned kernels give every (sequence, KV head, partition) its own
// CTA; for batches of many short contexts that means several waves of short
// CTAs, each paying a start-up and drain, and a last wave that leaves SMs
// idle.  Here the work is balanced instead: the tiles of all (sequence,
// KV head) segments, in order, form one sequence of N 16-token tiles, and
// consumer warp w of a single wave of CTAs streams tiles [w*Q, (w+1)*Q) with
// Q = ceil(N / warps).  A warp crosses segment boundaries without draining
// its pipeline; each segment piece it covers yields a partial result, and the
// last warp to finish a segment merges its pieces (log-sum-exp) into the
// output.  A one-CTA plan kernel first scans the per-sequence tile counts.
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
        const int T = prefix[b + 1] - prefix[b];
        const long long off = x - (long long)p.num_kv_heads * prefix[b];
        const int g = (int)(off / T);
        starts[ws] = make_int4(b, g, (int)(off - (long long)g * T), T);
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
struct BalancedLayout {
    static constexpr int kRing = kFp8 ? kStagesFp8 : kStages;
    static constexpr int kPerWarp = kRing / kConsumerWarps;       // stages per consumer warp
    static constexpr int kBoxBytes = kBox16Bytes;
    static constexpr int kHalves = kFp8 ? 1 : D / kBoxElems;
    static constexpr int kTileBytes = kHalves * kBoxBytes;
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kPipeBytes = kRing * kStageBytes;
    static constexpr int kTile16Bytes = (D / kBoxElems) * kBoxBytes;
    static constexpr int kConvBytes = kFp8 ? kConsumerWarps * 2 * kTile16Bytes : 0;
    static constexpr int kDynamicSmem = kPipeBytes + kConvBytes + 1024;
};

// Writes the fused step's new token (chunk c of K or V, head g) into the
// cache and returns it in the 16-bit compute type; FP8 caches get E4M3 codes.
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
    uint32_t back[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 f = Mma<T>::unpack(w[j]);
        q[j] = f32x2_to_e4m3x2(__fdiv_rn(f.y, sc), __fdiv_rn(f.x, sc));
        back[j] = e4m3x2_to<T>(q[j]);
    }
    uint8_t* cache = reinterpret_cast<uint8_t*>(is_k ? p.k_cache : p.v_cache);
    *reinterpret_cast<uint2*>(cache + dst + 8 * c) =
        make_uint2((uint32_t)q[0] | ((uint32_t)q[1] << 16), (uint32_t)q[2] | ((uint32_t)q[3] << 16));
    return make_uint4(back[0], back[1], back[2], back[3]);
}

// Log-sum-exp merge of the np pieces (records wfirst + j + z) of segment z by
// one warp: lanes take pieces for the maximum and the weights, then own D/32
// output dims each and sum the pieces, four records in flight.
template <typename T, int D>
__device__ __forceinline__ void merge_pieces(const BalancedParams& p, int z, long long wfirst,
                                             int np, size_t qh0, int G, int lane) {
    constexpr int V = D / 32;
    for (int h = 0; h < G; ++h) {
        float mx = -INFINITY;
        for (int j = lane; j < np; j += 32)
            mx = fmaxf(mx, __ldcg(p.rec_m + (size_t)(wfirst + j + z) * G + h));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float acc[V];
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.f;
        float den = 0.f;
        for (int j0 = 0; j0 < np; j0 += 32) {
            const int j = j0 + lane;
            float wj = 0.f;
            if (j < np) {
                const size_t r = (size_t)(wfirst + j + z);
                wj = __ldcg(p.rec_l + r * G + h) * ex2(__ldcg(p.rec_m + r * G + h) - mx);
            }
            den += wj;
            const int n = min(32, np - j0);
            for (int i = 0; i < n; i += 4) {
                float x[4][V], wt[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    wt[u] = __shfl_sync(0xffffffffu, wj, (i + u) & 31);
                    const size_t r = (size_t)(wfirst + j0 + min(i + u, n - 1) + z);
                    const float* src = p.rec_o + (r * G + h) * D + lane * V;
#pragma unroll
                    for (int e = 0; e < V; ++e) x[u][e] = __ldcg(src + e);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (i + u < n) {
#pragma unroll
                        for (int e = 0; e < V; ++e) acc[e] += wt[u] * x[u][e];
                    }
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        T* out = reinterpret_cast<T*>(p.out) + (qh0 + h) * D + lane * V;
#pragma unroll
        for (int e = 0; e < V; ++e) out[e] = from_float<T>(acc[e] / den);
    }
}

template <typename T, int D, bool kFp8>
__global__ void __launch_bounds__(kDecodeThreads, kFp8 ? kMinCtasPerSmFp8 : kMinCtasPerSm)
    balanced_step_kernel(const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v,
                         const __grid_constant__ BalancedParams p) {
    using Lay = BalancedLayout<D, kFp8>;
    using M = Mma<T>;
    static_assert(!kFp8 || D == 128, "the FP8 cache is built for head_dim 128");
    __shared__ __align__(8) uint64_t full_bar[Lay::kRing];
    __shared__ __align__(8) uint64_t empty_bar[Lay::kRing];
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int B = p.num_seqs, Hkv = p.num_kv_heads, G = p.group;

    grid_dependency_wait();                  // the plan and the inputs are ready
    allow_dependent_launch();
    const int* prefix = p.plan + 2;
    const long long N = p.plan[0];
    const int Q = p.plan[1];

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
        // producer: the W consumer streams' tiles, round robin, 32 at a time
        // ------------------------------------------------------------------
        if (lane == 0) {
            prefetch_tensor_map(&tmap_k);
            prefetch_tensor_map(&tmap_v);
        }
        const int tiles_per_block = p.block_size / kTileTokens;
        long long first[kConsumerWarps];
        int count[kConsumerWarps];
        TileCursor cur[kConsumerWarps];
        int maxcount = 0;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            const long long ws = (long long)blockIdx.x * kConsumerWarps + w;
            first[w] = ws * Q;
            count[w] = (int)max(0LL, min((long long)Q, N - first[w]));
            if (count[w] > 0) cur[w].load(p.plan, B, ws);
            maxcount = max(maxcount, count[w]);
        }
        // per stream: descriptors of the next 32 tiles, one per lane
        int blk[kConsumerWarps], gg[kConsumerWarps], sub[kConsumerWarps];
        bool ok = true;
        for (int k0 = 0; k0 < maxcount && ok; k0 += 32) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                blk[w] = 0, gg[w] = 0, sub[w] = 0;
                if (k0 < count[w]) {
                    TileCursor c = cur[w];
                    c.advance(lane, prefix, B, Hkv);
                    if (k0 + lane < count[w]) {
                        blk[w] = __ldg(p.block_tables + (size_t)c.b * p.max_blocks_per_seq +
                                       c.t / tiles_per_block);
                        if (blk[w] < 0 || blk[w] >= p.num_blocks)
                            flag_error(p.err, PA_DEVERR_BAD_CONTEXT);
                        gg[w] = c.g;
                        sub[w] = (c.t % tiles_per_block) * kTileTokens;
                    }
                    // the stream's cursor for the next batch: lane 31's position + 1
                    c.advance(1, prefix, B, Hkv);
                    cur[w].b = __shfl_sync(0xffffffffu, c.b, 31);
                    cur[w].g = __shfl_sync(0xffffffffu, c.g, 31);
                    cur[w].t = __shfl_sync(0xffffffffu, c.t, 31);
                    cur[w].T = __shfl_sync(0xffffffffu, c.T, 31);
                }
            }
            for (int j = 0; j < 32 && ok; ++j) {
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const int k = k0 + j;
                    const int pb = __shfl_sync(0xffffffffu, blk[w], j);
                    const int pg = __shfl_sync(0xffffffffu, gg[w], j);
                    const int ps = __shfl_sync(0xffffffffu, sub[w], j);
                    if (k >= count[w]) continue;
                    if (lane == 0) {
                        const int st = w + kConsumerWarps * (k % Lay::kPerWarp);
                        const int lap = k / Lay::kPerWarp;
                        if (lap > 0 && !mbar_wait(&empty_bar[st], (lap - 1) & 1)) {
                            flag_error(p.err, PA_DEVERR_WAIT_TIMEOUT);
                            ok = false;
                        } else {
                            mbar_arrive_expect_tx(&full_bar[st], Lay::kStageBytes);
                            uint8_t* kdst = smem + st * Lay::kStageBytes;
                            uint8_t* vdst = kdst + Lay::kTileBytes;
#pragma unroll
                            for (int hh = 0; hh < Lay::kHalves; ++hh) {
                                tma_load_4d(kdst + hh * Lay::kBoxBytes, &tmap_k, &full_bar[st],
                                            hh * kBoxElems, pg, ps, pb);
                                tma_load_4d(vdst + hh * Lay::kBoxBytes, &tmap_v, &full_bar[st],
                                            hh * kBoxElems, pg, ps, pb);
                            }
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                }
            }
        }
        return;
    }

    // ----------------------------------------------------------------------
    // consumer warp: its tile range, piece by piece
    // ----------------------------------------------------------------------
    const long long ws = (long long)blockIdx.x * kConsumerWarps + warp;
    const long long x0 = ws * Q;
    const int count = (int)max(0LL, min((long long)Q, N - x0));
    if (count == 0) return;
    const int max_ctx = p.max_blocks_per_seq * p.block_size;
    const int r8 = lane >> 2, c4 = lane & 3;
    const int hA = 2 * c4, hB = 2 * c4 + 1;
    uint8_t* conv = smem + Lay::kPipeBytes + warp * 2 * Lay::kTile16Bytes;

    TileCursor cur;
    cur.load(p.plan, B, ws);
    const T* qbase = reinterpret_cast<const T*>(p.q);
    uint32_t qb[D / 16][2], qn[D / 16][2];
    TileState<D> ts;
    // the first piece's query rows and length; later pieces' are prefetched
    // during the last tile of the piece before
    load_q_fragments<T, D>(qn, qbase + ((size_t)cur.b * p.num_q_heads + (size_t)cur.g * G) * D, G,
                           lane);
    int L_next = p.context_lens[cur.b];
    int L = 0;
    for (int k = 0; k < count; ++k) {
        const int b = cur.b, g = cur.g, t = cur.t;
        if (k == 0 || t == 0) {                          // a piece begins
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) qb[kk][0] = qn[kk][0], qb[kk][1] = qn[kk][1];
            L = L_next < 0 ? 0 : (L_next > max_ctx ? max_ctx : L_next);
            ts.reset();
        }
        const bool piece_end = (k == count - 1) || (t == cur.T - 1);
        if (piece_end && k + 1 < count) {
            // prefetch the next piece (the next segment) while this tile runs
            TileCursor nx = cur;
            nx.advance(1, prefix, B, Hkv);
            load_q_fragments<T, D>(qn, qbase + ((size_t)nx.b * p.num_q_heads + (size_t)nx.g * G) * D,
                                   G, lane);
            L_next = p.context_lens[nx.b];
        }
        const int st = warp + kConsumerWarps * (k % Lay::kPerWarp);
        bool ok = mbar_wait(&full_bar[st], (k / Lay::kPerWarp) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) flag_error(p.err, PA_DEVERR_WAIT_TIMEOUT);
            return;
        }
        uint8_t* ktile = smem + st * Lay::kStageBytes;
        uint8_t* vtile = ktile + Lay::kTileBytes;
        if (kFp8) {
            convert_fp8_tiles<T>(ktile, conv, conv + Lay::kTile16Bytes, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[st]);
            ktile = conv;
            vtile = conv + Lay::kTile16Bytes;
        }
        if (t == (L - 1) / kTileTokens) {
            // the segment's last tile holds its new token (position L - 1)
            const int64_t slot = p.slot_mapping[b];
            if (slot >= 0) {
                const int pos = L - 1;
                const int64_t blk = p.block_tables[(size_t)b * p.max_blocks_per_seq +
                                                   pos / p.block_size];
                if (slot == blk * p.block_size + pos % p.block_size && blk >= 0 &&
                    blk < p.num_blocks) {
                    const int c = lane & 15;
                    if (c < D / 8) {
                        const bool is_k = lane < 16;
                        put_tile_chunk(is_k ? ktile : vtile, pos % kTileTokens, c,
                                       balanced_new_token<T, D, kFp8>(p, b, g, slot, c, is_k));
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                } else if (lane == 0 && g == 0) {
                    flag_error(p.err, PA_DEVERR_BAD_SLOT);
                }
            }
        }
        attend_tile<T, D>(ts, qb, ktile, vtile, t * kTileTokens, L, p.scale_log2, lane);
        __syncwarp();
        if (!kFp8 && lane == 0) mbar_arrive(&empty_bar[st]);

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
                    const int d = 16 * n + r8;
                    if (hA < G) {
                        out[hA * D + d] = from_float<T>(ts.acc[n][0] * iA);
                        out[hA * D + d + 8] = from_float<T>(ts.acc[n][2] * iA);
                    }
                    if (hB < G) {
                        out[hB * D + d] = from_float<T>(ts.acc[n][1] * iB);
                        out[hB * D + d + 8] = from_float<T>(ts.acc[n][3] * iB);
                    }
                }
            } else {
                // partial record: normalised o, true max, sum at the true max (log2 units)
                const size_t rec = (size_t)(ws + z);
                float* ro = p.rec_o + rec * G * D;
#pragma unroll
                for (int n = 0; n < D / 16; ++n) {
                    const int d = 16 * n + r8;
                    if (hA < G) {
                        ro[hA * D + d] = ts.acc[n][0] * iA;
                        ro[hA * D + d + 8] = ts.acc[n][2] * iA;
                    }
                    if (hB < G) {
                        ro[hB * D + d] = ts.acc[n][1] * iB;
                        ro[hB * D + d + 8] = ts.acc[n][3] * iB;
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
    const int smem = BalancedLayout<D, kFp8>::kDynamicSmem;
    e = cudaFuncSetAttribute(balanced_step_kernel<T, D, kFp8>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_with_pdl(balanced_step_kernel<T, D, kFp8>, dim3(num_ctas),
                           dim3(kDecodeThreads), smem, stream, tmk, tmv, p);
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
