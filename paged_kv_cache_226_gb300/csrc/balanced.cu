// Work-balanced fused decode layer-step.
//
// The partitioned kernels give every (sequence, KV head, partition) its own
// CTA; for batches of many short contexts that means more than one wave of
// CTAs: the CTAs of the first wave end together and their successors ramp up
// together (a dip), and the CTAs that start last stream their partition with
// few neighbours at the end of the launch (a tail).  Here the work is
// balanced instead: the tiles of all (sequence, KV head) segments, in order,
// form one sequence of N 16-token tiles, and consumer warp w of a single wave
// of CTAs streams tiles [w*Q, (w+1)*Q) with Q = ceil(N / warps), so every
// warp runs from the start of the launch to its end.
//
// The CTA has the fused step's shape: a TMA producer warp and two consumer
// warps sharing one ring (stage s belongs to consumer s % 2), six CTAs per
// SM, one wave.  The producer walks both consumers' ranges, reading the
// block table a batch of 32 tiles ahead, and issues whichever consumer's
// next stage is free.  A consumer crosses segment boundaries without
// draining the ring; each segment piece it covers yields a partial result
// (or, for a whole segment, the output), and the last warp to finish a
// segment merges the pieces (log-sum-exp) into the output.  Every warp finds
// the start of its range itself, in one pass over the batch's context
// lengths, so no plan kernel runs before it.
//
// The cache write of the new token and its use by attention follow the
// fused step (pa_decode_step).
#include "decode_kernel.cuh"

namespace pa {

// A tile position no batch reaches.
constexpr long long kNever = 1LL << 62;

// Tiles of sequence b: its context, clamped to its table row, in 16-token tiles.
__device__ __forceinline__ int seq_tiles(const BalancedParams& p, int b, int max_ctx) {
    int L = __ldg(p.context_lens + b);
    L = L < 0 ? 0 : (L > max_ctx ? max_ctx : L);
    return (L + kTileTokens - 1) / kTileTokens;
}

// Position of a tile in the (sequence, KV head, tile) order.
struct TileCursor {
    int b, g, t, T;           // sequence, KV head, tile within the segment, tiles of b

    // Moves n >= 0 tiles forward (stops at the end of the batch).
    __device__ __forceinline__ void advance(int n, const BalancedParams& p, int B, int Hkv,
                                            int max_ctx) {
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
                    T = seq_tiles(p, b, max_ctx);
                } while (T == 0);
            }
        }
    }
};

// A warp-wide pass over the context lengths: the total tile count N (all KV
// heads) and, for each of K positions x[i] < N, the cursor of that tile
// (positions >= N are never found).  Segment z = b * Hkv + g starts at tile
// Hkv * prefix_b + g * T_b, prefix_b being the tiles of the sequences before
// b.  With stop_when_found the pass ends as soon as every position is found,
// and the returned total is then incomplete.
template <int K>
__device__ __forceinline__ long long locate(const BalancedParams& p, int B, int Hkv, int max_ctx,
                                            int lane, const long long (&x)[K],
                                            TileCursor (&cur)[K], bool stop_when_found) {
    long long run = 0;                       // tiles per head of the sequences before this chunk
    bool found[K];
#pragma unroll
    for (int i = 0; i < K; ++i) found[i] = false;
    for (int base = 0; base < B; base += 32) {
        const int b = base + lane;
        const int T = b < B ? seq_tiles(p, b, max_ctx) : 0;
        int incl = T;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const long long excl = run + incl - T;
#pragma unroll
        for (int i = 0; i < K; ++i) {
            if (found[i]) continue;
            const unsigned m = __ballot_sync(0xffffffffu, (long long)Hkv * (run + incl) > x[i]);
            if (m != 0u) {
                const int l = __ffs(m) - 1;
                const int Tl = __shfl_sync(0xffffffffu, T, l);
                const long long ex = __shfl_sync(0xffffffffu, excl, l);
                const long long off = x[i] - (long long)Hkv * ex;
                cur[i].b = base + l;
                cur[i].g = (int)(off / Tl);
                cur[i].t = (int)(off - (long long)cur[i].g * Tl);
                cur[i].T = Tl;
                found[i] = true;
            }
        }
        run += __shfl_sync(0xffffffffu, incl, 31);
        if (stop_when_found) {
            bool all = true;
#pragma unroll
            for (int i = 0; i < K; ++i) all = all && found[i];
            if (all) break;
        }
    }
    return run * Hkv;
}

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
// one warp, four heads of the group at a time.  Lanes take pieces for the
// per-head maxima and weights; for the weighted sum each lane owns D/32 dims
// of each of the four heads and keeps two pieces' worth of loads in flight.
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
    constexpr int kH = 4;                         // heads per pass
    for (int h0 = 0; h0 < G; h0 += kH) {
        float mx[kH], den[kH], acc[kH][V];
#pragma unroll
        for (int h = 0; h < kH; ++h) {
            mx[h] = -INFINITY;
            den[h] = 0.f;
#pragma unroll
            for (int e = 0; e < V; ++e) acc[h][e] = 0.f;
        }
        for (int j = lane; j < np; j += 32) {
            const size_t r = (size_t)(wfirst + j + z) * G + h0;
#pragma unroll
            for (int h = 0; h < kH; ++h)
                if (h0 + h < G) mx[h] = fmaxf(mx[h], __ldcg(p.rec_m + r + h));
        }
#pragma unroll
        for (int h = 0; h < kH; ++h) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], o));
        }
        for (int j0 = 0; j0 < np; j0 += 32) {
            const int j = j0 + lane;
            float w[kH];
#pragma unroll
            for (int h = 0; h < kH; ++h) w[h] = 0.f;
            if (j < np) {
                const size_t r = (size_t)(wfirst + j + z) * G + h0;
#pragma unroll
                for (int h = 0; h < kH; ++h)
                    if (h0 + h < G)
                        w[h] = __ldcg(p.rec_l + r + h) * ex2(__ldcg(p.rec_m + r + h) - mx[h]);
            }
#pragma unroll
            for (int h = 0; h < kH; ++h) den[h] += w[h];
            const int n = min(32, np - j0);
            for (int i = 0; i < n; i += 2) {
                float x[2][kH][V];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const size_t r = (size_t)(wfirst + j0 + min(i + u, n - 1) + z) * G + h0;
                    const float* src = p.rec_o + r * D + lane * V;
#pragma unroll
                    for (int h = 0; h < kH; ++h)
                        if (h0 + h < G) load_vec<V>(x[u][h], src + h * D);
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (i + u < n) {
#pragma unroll
                        for (int h = 0; h < kH; ++h) {
                            if (h0 + h < G) {
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
        for (int h = 0; h < kH; ++h) {
            if (h0 + h < G) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    den[h] += __shfl_xor_sync(0xffffffffu, den[h], o);
                T* out = reinterpret_cast<T*>(p.out) + (qh0 + h0 + h) * D + lane * V;
#pragma unroll
                for (int e = 0; e < V; ++e) out[e] = from_float<T>(acc[h][e] / den[h]);
            }
        }
    }
}

template <typename T, int D, bool kFp8>
__global__ void __launch_bounds__(kDecodeThreads, kFp8 ? kMinCtasPerSmFp8 : kMinCtasPerSm)
    balanced_step_kernel(const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v,
                         const __grid_constant__ BalancedParams p) {
    using Lay = DecodeLayout<D, kFp8>;
    constexpr int R = Lay::kRing;
    constexpr int kPer = R / kConsumerWarps;          // stages of one consumer
    static_assert(!kFp8 || D == 128, "the FP8 cache is built for head_dim 128");
    __shared__ __align__(8) uint64_t full_bar[R];
    __shared__ __align__(8) uint64_t empty_bar[R];
    __shared__ int4 pend_smem[kConsumerWarps][2];
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // barriers and tensor maps before the inputs are ready
    if (threadIdx.x == 0) {
        for (int s = 0; s < R; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        fence_barrier_init();
    }
    if (warp == kConsumerWarps && lane == 0) {
        prefetch_tensor_map(&tmap_k);
        prefetch_tensor_map(&tmap_v);
    }
    __syncthreads();
    grid_dependency_wait();                  // the inputs are ready
    allow_dependent_launch();

    const int B = p.num_seqs, Hkv = p.num_kv_heads, G = p.group;
    const int max_ctx = p.max_blocks_per_seq * p.block_size;
    const int tiles_per_block = p.block_size / kTileTokens;
    const long long first_ws = (long long)blockIdx.x * kConsumerWarps;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------------
        // producer: both consumers' ranges -> TMA boxes
        // ------------------------------------------------------------------
        long long x[kConsumerWarps];
        TileCursor bc[kConsumerWarps];
#pragma unroll
        for (int c = 0; c < kConsumerWarps; ++c) x[c] = kNever;
        // first pass: N only (positions unknown until Q is)
        const long long N = locate<kConsumerWarps>(p, B, Hkv, max_ctx, lane, x, bc, false);
        const long long Q = max(1LL, (N + p.num_warps - 1) / p.num_warps);
        int count[kConsumerWarps];
#pragma unroll
        for (int c = 0; c < kConsumerWarps; ++c) {
            const long long x0 = (first_ws + c) * Q;
            count[c] = (int)max(0LL, min(Q, N - x0));
            x[c] = count[c] > 0 ? x0 : kNever;
        }
        if (count[0] == 0 && count[1] == 0) return;
        (void)locate<kConsumerWarps>(p, B, Hkv, max_ctx, lane, x, bc, true);
        // descriptors (block, KV head, token offset) of 32 tiles at a time,
        // one per lane: set A is the batch being issued, set B the next one,
        // whose table reads have 32 issues' time to land
        int a_blk[kConsumerWarps], a_g[kConsumerWarps], a_sub[kConsumerWarps];
        int b_blk[kConsumerWarps], b_g[kConsumerWarps], b_sub[kConsumerWarps];
        auto describe = [&](int c, int i0, int& blk, int& gg, int& sub) {
            blk = 0, gg = 0, sub = 0;
            if (i0 >= count[c]) return;
            TileCursor cc = bc[c];
            cc.advance(lane, p, B, Hkv, max_ctx);
            if (i0 + lane < count[c]) {
                blk = __ldg(p.block_tables + (size_t)cc.b * p.max_blocks_per_seq +
                            cc.t / tiles_per_block);
                gg = cc.g;
                sub = (cc.t % tiles_per_block) * kTileTokens;
            }
            cc.advance(1, p, B, Hkv, max_ctx);
            bc[c].b = __shfl_sync(0xffffffffu, cc.b, 31);
            bc[c].g = __shfl_sync(0xffffffffu, cc.g, 31);
            bc[c].t = __shfl_sync(0xffffffffu, cc.t, 31);
            bc[c].T = __shfl_sync(0xffffffffu, cc.T, 31);
        };
#pragma unroll
        for (int c = 0; c < kConsumerWarps; ++c) {
            describe(c, 0, a_blk[c], a_g[c], a_sub[c]);
            describe(c, 32, b_blk[c], b_g[c], b_sub[c]);
        }
        // Issue whichever consumer's next stage is free, so that a consumer
        // that stops (a new piece's query rows, a record write) holds up
        // only its own stream.
        int next[kConsumerWarps];
#pragma unroll
        for (int c = 0; c < kConsumerWarps; ++c) next[c] = 0;
        uint64_t idle_since = 0;
        while (next[0] < count[0] || next[1] < count[1]) {
            bool progressed = false;
#pragma unroll
            for (int c = 0; c < kConsumerWarps; ++c) {
                const int k = next[c];
                if (k >= count[c]) continue;
                const int st = c + kConsumerWarps * (k % kPer);
                int free_ = 1;
                if (lane == 0 && k >= kPer)
                    free_ = mbar_test_wait(&empty_bar[st], ((k / kPer) - 1) & 1);
                if (!__shfl_sync(0xffffffffu, free_, 0)) continue;
                const int blk = __shfl_sync(0xffffffffu, a_blk[c], k & 31);
                const int gg = __shfl_sync(0xffffffffu, a_g[c], k & 31);
                const int sub = __shfl_sync(0xffffffffu, a_sub[c], k & 31);
                if (lane == 0) {
                    if (blk < 0 || blk >= p.num_blocks) flag_error(p.err, PA_DEVERR_BAD_CONTEXT);
                    uint8_t* kdst = smem + st * Lay::kStageBytes;
                    uint8_t* vdst = kdst + Lay::kTileBytes;
                    mbar_arrive_expect_tx(&full_bar[st], Lay::kStageBytes);
#pragma unroll
                    for (int hh = 0; hh < Lay::kHalves; ++hh) {
                        tma_load_4d(kdst + hh * Lay::kBoxBytes, &tmap_k, &full_bar[st],
                                    hh * kBoxElems, gg, sub, blk);
                        tma_load_4d(vdst + hh * Lay::kBoxBytes, &tmap_v, &full_bar[st],
                                    hh * kBoxElems, gg, sub, blk);
                    }
                }
                next[c] = k + 1;
                progressed = true;
                if (((k + 1) & 31) == 0 && k + 1 < count[c]) {
                    a_blk[c] = b_blk[c], a_g[c] = b_g[c], a_sub[c] = b_sub[c];
                    describe(c, k + 1 + 32, b_blk[c], b_g[c], b_sub[c]);
                }
            }
            if (progressed) {
                idle_since = 0;
            } else {
                // both consumers' next stages are busy: back off briefly; a
                // stage that stays busy past the wait limit is an error
                const uint64_t now = global_timer_ns();
                if (idle_since == 0) {
                    idle_since = now;
                } else if (now - idle_since > kWaitLimitNs) {
                    if (lane == 0) flag_error(p.err, PA_DEVERR_WAIT_TIMEOUT);
                    return;
                }
                __nanosleep(64);
            }
        }
        return;
    }

    // ----------------------------------------------------------------------
    // consumers: attention over the warp's range, piece by piece
    // ----------------------------------------------------------------------
    const long long ws = first_ws + warp;

    // sequences with nothing to attend (empty or negative context): zero
    // output, and a new token for them is an error; each is handled by one
    // warp of the grid
    for (long long b = ws; b < B; b += p.num_warps) {
        const int Lraw = p.context_lens[b];
        if (Lraw < 0 || Lraw > max_ctx) {
            if (lane == 0) flag_error(p.err, PA_DEVERR_BAD_CONTEXT);
        }
        if (Lraw <= 0) {
            T* out = reinterpret_cast<T*>(p.out) + (size_t)b * p.num_q_heads * D;
            for (int i = lane; i < p.num_q_heads * D; i += 32) out[i] = from_float<T>(0.f);
            if (lane == 0 && p.slot_mapping[b] >= 0) flag_error(p.err, PA_DEVERR_BAD_SLOT);
        }
    }

    long long x[1] = {kNever};
    TileCursor cur1[1];
    const long long N = locate<1>(p, B, Hkv, max_ctx, lane, x, cur1, false);
    const long long Q = max(1LL, (N + p.num_warps - 1) / p.num_warps);
    const long long x0 = ws * Q;
    const int count = (int)max(0LL, min(Q, N - x0));
    if (count == 0) return;
    x[0] = x0;
    (void)locate<1>(p, B, Hkv, max_ctx, lane, x, cur1, true);
    TileCursor cur = cur1[0];
    const int r8 = lane >> 2, c4 = lane & 3;
    const int hA = 2 * c4, hB = 2 * c4 + 1;

    const T* qbase = reinterpret_cast<const T*>(p.q);
    uint32_t qb[D / 16][2];
    TileState<D> ts;
    // The query rows of the group are read when a piece begins; the next
    // piece's rows (G x D contiguous 16-bit values) are prefetched into L1
    // during the last tile of the piece before, so that read finds them.
    auto prefetch_q = [&](const TileCursor& c) {
        const char* src = reinterpret_cast<const char*>(
            qbase + ((size_t)c.b * p.num_q_heads + (size_t)c.g * G) * D);
        if (lane * 128 < G * D * (int)sizeof(T))
            asm volatile("prefetch.global.L1 [%0];" ::"l"(src + lane * 128));
    };
    // segments this warp finishes last (at most two: only its first and last
    // pieces can be shared with other warps), merged after the range;
    // kept in shared memory, off the loop's registers
    int4* pend = pend_smem[warp];
    if (lane < 2) pend[lane] = make_int4(-1, 0, 0, 0);
    __syncwarp();
    float scale_log2 = p.scale_log2;
    int L_next = p.context_lens[cur.b];
    int64_t slot_next = p.slot_mapping[cur.b];
    int L = 0;
    int64_t slot = -1;
    for (int k = 0; k < count; ++k) {
        const int b = cur.b, g = cur.g, t = cur.t;
        if (k == 0 || t == 0) {                          // a piece begins
            const T* qg = qbase + ((size_t)b * p.num_q_heads + (size_t)g * G) * D;
            if constexpr (kFp8) {
                const int sq = load_q_fragments_fp8<T>(qb, qg, G, lane);   // q / 2^sq in fp16
                scale_log2 = p.scale_log2 * __int_as_float((127 + sq) << 23);
            } else {
                load_q_fragments<T, D>(qb, qg, G, lane);
            }
            L = L_next < 0 ? 0 : (L_next > max_ctx ? max_ctx : L_next);
            slot = slot_next;
            ts.reset();
        }
        const bool piece_end = (k == count - 1) || (t == cur.T - 1);
        if (piece_end && k + 1 < count) {
            TileCursor nx = cur;
            nx.advance(1, p, B, Hkv, max_ctx);
            prefetch_q(nx);
            L_next = p.context_lens[nx.b];
            slot_next = p.slot_mapping[nx.b];
        }
        const int st = warp + kConsumerWarps * (k % kPer);
        bool ok = mbar_wait(&full_bar[st], (k / kPer) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) flag_error(p.err, PA_DEVERR_WAIT_TIMEOUT);
            return;
        }
        uint8_t* ktile = smem + st * Lay::kStageBytes;
        uint8_t* vtile = ktile + Lay::kTileBytes;
        if (slot >= 0 && t == (L - 1) / kTileTokens) {
            // the segment's last tile holds its new token (position L - 1)
            const int pos = L - 1;
            const int64_t blk = __ldg(p.block_tables + (size_t)b * p.max_blocks_per_seq +
                                      pos / p.block_size);
            if (slot == blk * p.block_size + pos % p.block_size && blk >= 0 &&
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
            // the codes are in registers: the stage can be refilled
            attend_tile_fp8(ts, [&](int kk, uint32_t& b0, uint32_t& b1) { b0 = qb[kk][0]; b1 = qb[kk][1]; },
                            ktile, vtile, t * kTileTokens, L, scale_log2, lane,
                            [&] { release_stage(&empty_bar[st], lane); });
        } else {
            attend_tile<T, D>(ts, [&](int kk, uint32_t& b0, uint32_t& b1) { b0 = qb[kk][0]; b1 = qb[kk][1]; },
                              ktile, vtile, t * kTileTokens, L, scale_log2, lane);
            release_stage(&empty_bar[st], lane);
        }

        if (piece_end) {
            ts.reduce_row_sums();
            const int z = b * Hkv + g;
            const long long s0 = x0 + k - t;             // the segment's first tile
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
                // partial record: normalised o, true max, sum at the true max
                // (log2 units); record ws + z is unique, since a later warp
                // covers only the same or later segments
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
                // the warp sync orders the lanes' record writes before lane 0's
                // acq_rel add (release); the add that completes the segment
                // acquires every other piece's records for this warp
                __syncwarp();
                int last = 0;
                if (lane == 0) {
                    int before;
                    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                                 : "=r"(before)
                                 : "l"(p.counters + z)
                                 : "memory");
                    last = before == (int)(wlast - wfirst);
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    // the merge waits for the end of the range, when the
                    // accumulators are dead (a segment's last piece to finish
                    // is almost always at the end of some warp's range anyway)
                    if (lane == 0)
                        pend[pend[0].x < 0 ? 0 : 1] = make_int4(
                            z, (int)(wlast - wfirst + 1), (int)(wfirst & 0xffffffff),
                            (int)(wfirst >> 32));
                    __syncwarp();
                }
            }
        }
        cur.advance(1, p, B, Hkv, max_ctx);
    }
    __syncwarp();
    for (int i = 0; i < 2; ++i) {
        const int4 e = pend[i];
        if (e.x < 0) continue;
        const int z = e.x, b = z / Hkv, g = z - b * Hkv;
        const long long wfirst = (long long)(unsigned)e.z | ((long long)e.w << 32);
        merge_pieces<T, D>(p, z, wfirst, e.y, (size_t)b * p.num_q_heads + (size_t)g * G, G, lane);
        if (lane == 0) p.counters[z] = 0;
    }
}

template <typename T, int D, bool kFp8>
cudaError_t launch_balanced_t(const CUtensorMap& tmk, const CUtensorMap& tmv,
                              const BalancedParams& p, int num_ctas, cudaStream_t stream) {
    // this kernel holds its q fragments in registers: no q area
    const int smem = DecodeLayout<D, kFp8>::kDynamicSmem - DecodeLayout<D, kFp8>::kQBytes;
    cudaError_t e = cudaFuncSetAttribute(balanced_step_kernel<T, D, kFp8>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = launch_with_pdl(balanced_step_kernel<T, D, kFp8>, dim3(num_ctas), dim3(kDecodeThreads),
                        smem, stream, tmk, tmv, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
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
