// Chunked-prefill attention on the fifth-generation tensor cores (tcgen05,
// tensor-memory accumulators), head_dim 128 and GQA groups of 1, 2, 4 or 8.
//
// Sequence b holds L_b tokens, the last C_b of which are new; new token i
// sits at position L_b - C_b + i and attends causally to positions 0..itself
// (ta-paperlens page, prefill vs decode and the quadratic cost of prefill;
// techfeed summary, chunked prefill).  A unit of work is 128 query rows: 128
// / G new tokens of one (sequence, KV head) times the G query heads that read
// that KV head, so every K/V tile is read once for all of them.  One
// persistent CTA per SM walks its units (a snake over the schedule, longest
// first); its rings, tensor-memory buffers and barriers run on from one unit
// to the next, so that the next unit's copies, Q and first S products
// overlap the end of the current one (many short units: 266 -> 218 us
// against a CTA per unit).
//
// Per 128-key tile j (keys 128 j .. 128 j + 127 through the block table):
//   S_j = Q K_j^T          128 x 128 x 128 into tensor memory (three
//                          buffers), Q from shared memory (stored there once,
//                          laid out like a K tile), K from its TMA-staged tile
//   P_j = 2^(S_j - m)      four softmax warps, one thread per row (all 128
//                          keys of the tile), a lazily raised running max m (log2
//                          units, threshold 2^8: the accumulator is rescaled
//                          in tensor memory only when a row's max grows by
//                          more than that); P goes to tensor memory over S_j
//                          (already in registers; bf16: a hi and a lo part
//                          cut from the fp32 bits, together exact to 2^-15)
//   O  += P_j V_j          128 x 128 x 128, P read from tensor memory, V from
//                          its TMA-staged [key][dim] tile (MN-major), O in
//                          tensor memory
// Warp roles: warp 0 streams K tiles and warp 6 V tiles (three and two
// stages beside Q in shared memory) with TMA, 16-token boxes of the paged
// cache, each at its own pace; lane 0 of warp 1 issues the S products and
// lane 0 of warp 7 the P V products, committing them to mbarriers; warps
// 2-5 run the softmax and the epilogue.  One control warp and one softmax
// warp sit on each of the SM's four schedulers: a thread issuing MMAs beside
// warps with ALU work ready is starved of issue slots, and two issuers halve
// what each must get through.  S_{j+1} and S_{j+2} are issued before P_j is ready, and P_j is
// computed and stored before P_{j-1} V_{j-1} has finished (only a rescale of O
// waits for that product); S_{j+3} overwrites P_j, so its issuer waits for
// P_j V_j first.  The P-ready barrier is kept per buffer too: the softmax may
// run two tiles ahead of the P V issuer, and one barrier would let its phases
// pass the issuer's parity check.
// Every mbarrier wait gives up after 1 s and flags PA_DEVERR_WAIT_TIMEOUT;
// the softmax warps then run their remaining iterations without waiting (so
// their barriers always complete), and tensor memory is always released.
#include "decode_tile.cuh"
#include "prefill_internal.h"
#include "tc_device.cuh"

namespace pa {

// bf16 P as a hi + lo pair (two P V products) or rounded once to bf16
#ifndef PA_PREFILL_SPLIT_P
#define PA_PREFILL_SPLIT_P 1
#endif

constexpr int kTcRows = 128;                 // query rows per CTA (tokens x heads)
constexpr int kTcKeys = 128;                 // keys per K/V tile
constexpr int kTcKStages = 3;                // K tiles in flight (free once S is computed)
constexpr int kTcVStages = 2;                // V tiles in flight (held until P V is done)
constexpr int kTcSBufs = 3;                  // S / P buffers in tensor memory
// one softmax thread per query row (all 128 keys of a tile; four softmax
// warps, one per scheduler beside the control warp) measured 4 % faster than
// two threads per row with maxima and sums exchanged through shared memory,
// which was 3 % faster than four: fewer ALU-ready warps beside the MMA issuers
constexpr int kTcChunks = 4;                 // 32-column tensor-memory accesses of a row
constexpr int kTcSoftmaxWarps = 4;
constexpr int kTcVWarp = 2 + kTcSoftmaxWarps;  // the V producer, after the softmax warps
constexpr int kTcPvWarp = 3 + kTcSoftmaxWarps; // issues P V (warp 1 issues S)
constexpr int kTcThreads = (4 + kTcSoftmaxWarps) * 32;
constexpr uint32_t kTcCols = 512;            // tensor-memory columns: S0/P0, S1/P1, S2/P2, O
constexpr int kTcOperand = 32768;            // 128 rows x 2 halves x 128 B
constexpr int kTcHalf = 16384;               // one 64-element half: 128 rows x 128 B

struct TcLayout {
    static constexpr int kQ = 0;             // two Q buffers: the current unit's and the next
    static constexpr int kK = kQ + 2 * kTcOperand;
    static constexpr int kV = kK + kTcKStages * kTcOperand;
    static constexpr int kBytes = kV + kTcVStages * kTcOperand;
    static constexpr int kDynamicSmem = kBytes + 1024;
    // with the few hundred bytes of static shared memory (barriers) this must
    // stay within the 227 KB a CTA may hold
    static_assert(kDynamicSmem + 512 <= 232448, "shared memory over the per-CTA limit");
};

// Byte offset of 16-byte chunk c (elements 8c .. 8c+7 of 128) of row r in an
// operand of two 64-element halves with the 128-byte swizzle.
__device__ __forceinline__ int tc_chunk(int r, int c) {
    return (c >> 3) * kTcHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// One unit of work: a (sequence, chunk) item of the schedule for one KV head.
struct TcUnit {
    int b, g;                // sequence, KV head
    int L, C, q0;            // context length, new tokens, first new token's row in q
    int t0, rows;            // first new token of the chunk, its tokens here
    int n_tiles;             // key tiles read: through the chunk's last position
};

template <typename T>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v,
                            const __grid_constant__ PrefillParams p) {
    constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr bool kSplitP = kBf16 && PA_PREFILL_SPLIT_P;
    using Lay = TcLayout;
    using M = Mma<T>;
    __shared__ __align__(8) uint64_t k_full[kTcKStages], k_empty[kTcKStages];
    __shared__ __align__(8) uint64_t v_full[kTcVStages], v_empty[kTcVStages];
    __shared__ __align__(8) uint64_t s_full[kTcSBufs], p_full[kTcSBufs], o_done[kTcSBufs];
    __shared__ __align__(8) uint64_t q_full[2];
    __shared__ uint32_t tmem_base;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group;
    const int QT = kTcRows / G;                             // new tokens per unit
    const int num_kv_heads = p.num_q_heads / G;
    const int n_items = p.num_seqs * p.max_chunks;
    const int n_units = n_items * num_kv_heads;
    const int max_ctx = p.max_blocks_per_seq * p.block_size;

    grid_dependency_wait();
    allow_dependent_launch();
    // The schedule's units are (item rank, KV head), heads fastest, longest
    // item first.  CTA c takes position c of even rounds of gridDim.x units
    // and position gridDim.x - 1 - c of odd rounds: a snake over the sorted
    // work, so that the CTAs' totals stay close.  Every role walks the same
    // units in the same order.
    auto unit_at = [&](int k, TcUnit& U) -> bool {
        const int c = (k & 1) ? (int)gridDim.x - 1 - (int)blockIdx.x : (int)blockIdx.x;
        const int u = k * (int)gridDim.x + c;
        if (u >= n_units) return false;
        U.g = u % num_kv_heads;
        const int rank = u / num_kv_heads;
        const int item = p.sched ? p.sched[rank] : n_items - 1 - rank;
        if (item < 0) return false;
        U.b = item / p.max_chunks;
        const int qt = item % p.max_chunks;
        const bool report = threadIdx.x == 0 && qt == 0 && U.g == 0;
        int L = p.context_lens[U.b];
        if (L < 0 || L > max_ctx) {
            if (report) flag_error(p.err, PA_DEVERR_BAD_CONTEXT);
            L = L < 0 ? 0 : max_ctx;
        }
        U.q0 = p.query_start[U.b];
        int C = p.query_start[U.b + 1] - U.q0;
        if (C > L) {
            if (report) flag_error(p.err, PA_DEVERR_BAD_CONTEXT);
            C = L;
        }
        U.L = L, U.C = C;
        U.t0 = qt * QT;
        if (U.t0 >= C) return false;
        U.rows = min(QT, C - U.t0);
        U.n_tiles = (L - C + U.t0 + U.rows - 1) / kTcKeys + 1;
        return true;
    };
    const int rounds = (n_units + (int)gridDim.x - 1) / (int)gridDim.x;

    // one operand (K or V) of tile j of unit U into stage gt % stages (gt:
    // the CTA's running tile count), 16-token boxes through the block table;
    // boxes wholly past the context are not loaded
    auto load = [&](const CUtensorMap* map, uint64_t* full, uint64_t* empty, int kind_off,
                    int stages, int gt, const TcUnit& U, int j) -> bool {
        const int32_t* table = p.block_tables + (size_t)U.b * p.max_blocks_per_seq;
        const int key0 = j * kTcKeys;
        const int nbox = min(8, (U.L - key0 + 15) / 16);
        int blk = 0, sub = 0;
        if (lane < nbox) {
            const int tok = key0 + 16 * lane;
            blk = __ldg(table + tok / p.block_size);
            sub = tok % p.block_size;
        }
        const int s = gt % stages;
        bool ok = true;
        if (lane == 0) {
            if (gt >= stages && !mbar_wait(&empty[s], ((gt / stages) - 1) & 1)) {
                flag_error(p.err, PA_DEVERR_WAIT_TIMEOUT);
                ok = false;
            } else {
                mbar_arrive_expect_tx(&full[s], (uint32_t)nbox * 2u * kBox16Bytes);
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) return false;
        if (lane < nbox && (blk < 0 || blk >= p.num_blocks)) flag_error(p.err, PA_DEVERR_BAD_CONTEXT);
        // lane i issues box i's two halves itself (the bytes to expect were
        // registered by lane 0 above, earlier in this warp's program order)
        uint8_t* dst = smem + kind_off + s * kTcOperand;
        if (lane < nbox) {
            tma_load_4d(dst + lane * kBox16Bytes, map, &full[s], 0, U.g, sub, blk);
            tma_load_4d(dst + kTcHalf + lane * kBox16Bytes, map, &full[s], kBoxElems, U.g, sub, blk);
        }
        return true;
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcKStages; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kTcVStages; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int i = 0; i < kTcSBufs; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], kTcSoftmaxWarps);         // one arrival per softmax warp
            mbar_init(&o_done[i], 1);
        }
        for (int i = 0; i < 2; ++i) mbar_init(&q_full[i], kTcSoftmaxWarps);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base, kTcCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base;
    const uint32_t tO = tmem + 128 * kTcSBufs;             // S_j / P_j in columns 128 (j % 3)

    if (warp == 0 || warp == kTcVWarp) {
        // ------------------------------------------------------------------
        // producers: K tiles (warp 0, free once S is computed, three stages)
        // and V tiles (warp 6, held until P V is done, two stages), each at
        // its own pace and on into the next unit's tiles
        // ------------------------------------------------------------------
        if (lane == 0) prefetch_tensor_map(warp == 0 ? &tmap_k : &tmap_v);
        bool ok = true;
        int gt = 0;
        for (int k = 0; k < rounds && ok; ++k) {
            TcUnit U;
            if (!unit_at(k, U)) continue;
            for (int j = 0; j < U.n_tiles && ok; ++j, ++gt) {
                ok = warp == 0 ? load(&tmap_k, k_full, k_empty, Lay::kK, kTcKStages, gt, U, j)
                               : load(&tmap_v, v_full, v_empty, Lay::kV, kTcVStages, gt, U, j);
            }
        }
    } else if (warp == 1 || warp == kTcPvWarp) {
        // ------------------------------------------------------------------
        // MMA issuers, one thread each on two schedulers: warp 1 issues S_j,
        // warp 7 P_j V_j, over the CTA's running tile count.  S_j overwrites
        // P_{j-3}, so it waits for that product (o_done of buffer j % 3); P V
        // in order accumulates O, each unit's first product overwriting it.
        // ------------------------------------------------------------------
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_f16(kTcRows, kTcKeys, kBf16, false);
            constexpr uint32_t kIdPV = idesc_f16(kTcRows, 128, kBf16, true);
            bool ok = true;
            int gt = 0, nu = 0;                             // tiles and units so far
            for (int k = 0; k < rounds && ok; ++k) {
                TcUnit U;
                if (!unit_at(k, U)) continue;
                if (warp == 1) {
                    // the unit's Q, in buffer nu % 2
                    const int qb = nu & 1;
                    ok = mbar_wait(&q_full[qb], (nu >> 1) & 1);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const uint32_t aQ = smem_u32(smem + Lay::kQ + qb * kTcOperand);
                    for (int j = 0; j < U.n_tiles; ++j, ++gt) {
                        const int s = gt % kTcKStages, sb = gt % kTcSBufs;
                        ok = mbar_wait(&k_full[s], (gt / kTcKStages) & 1);
                        if (ok && gt >= kTcSBufs) ok = mbar_wait(&o_done[sb], (gt / kTcSBufs - 1) & 1);
                        if (!ok) break;
                        tc_fence_after_sync();
                        const uint32_t aK = smem_u32(smem + Lay::kK + s * kTcOperand);
                        const uint32_t dS = tmem + 128 * sb;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint32_t off = (kk >> 2) * kTcHalf + (kk & 3) * 32;
                            mma_f16_ss(dS, smem_desc_sw128(aQ + off, 16, 1024),
                                       smem_desc_sw128(aK + off, 16, 1024), kIdS, kk > 0);
                        }
                        mma_commit(&s_full[sb]);
                        mma_commit(&k_empty[s]);            // S_j has read K_j
                    }
                } else {
                    for (int j = 0; j < U.n_tiles; ++j, ++gt) {
                        const int s = gt % kTcVStages, sb = gt % kTcSBufs;
                        ok = mbar_wait(&p_full[sb], (gt / kTcSBufs) & 1);
                        if (ok) ok = mbar_wait(&v_full[s], (gt / kTcVStages) & 1);
                        if (!ok) break;
                        tc_fence_after_sync();
                        const uint32_t aV = smem_u32(smem + Lay::kV + s * kTcOperand);
                        const uint32_t tP = tmem + 128 * sb;    // P_j over S_j
#pragma unroll
                        for (int part = 0; part < (kSplitP ? 2 : 1); ++part) {
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk)
                                mma_f16_ts(tO, tP + 64 * part + 8 * kk,
                                           smem_desc_sw128(aV + kk * 16 * 128, kTcHalf, 1024), kIdPV,
                                           j > 0 || part > 0 || kk > 0);
                        }
                        mma_commit(&o_done[sb]);
                        mma_commit(&v_empty[s]);            // P_j V_j has read V_j
                    }
                }
                ++nu;
            }
            if (!ok) flag_error(p.err, PA_DEVERR_WAIT_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------------
        // softmax and epilogue: this thread owns row r (tensor-memory lane r)
        // of every unit: all 128 keys of each tile and all 128 output dims
        // ------------------------------------------------------------------
        const int r = (warp & 3) * 32 + lane;
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const float sl = p.scale_log2;
        bool failed = false;                 // a wait ran out: finish the loops without waiting
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (!failed && !__all_sync(0xffffffffu, mbar_wait(bar, parity))) failed = true;
        };
        // this row of unit U's Q (zero past the chunk) into Q buffer `qb`,
        // laid out like a K tile, then visible to the tensor cores
        auto store_q = [&](const TcUnit& U, int qb) {
            const int t = r / G, h = r % G;
            const uint4* src = reinterpret_cast<const uint4*>(
                reinterpret_cast<const T*>(p.q) +
                ((size_t)(U.q0 + U.t0 + min(t, U.rows - 1)) * p.num_q_heads + (size_t)U.g * G + h) * 128);
            uint4 v[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) v[c] = t < U.rows ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
            uint8_t* dst = smem + Lay::kQ + qb * kTcOperand;
#pragma unroll
            for (int c = 0; c < 16; ++c) *reinterpret_cast<uint4*>(dst + tc_chunk(r, c)) = v[c];
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_full[qb]);
        };
        int k = 0, gt = 0, nu = 0;                          // round, tiles and units so far
        TcUnit U;
        bool have = false;
        for (; k < rounds && !have; ++k) have = unit_at(k, U);
        if (have) store_q(U, 0);
        while (have) {
            const int t = r / G, h = r % G;
            const int pos = min(U.L - U.C + U.t0 + t, U.L - 1);
            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < U.n_tiles; ++j, ++gt) {
                const int sv = gt % kTcVStages, sb = gt % kTcSBufs;
                const uint32_t tS = tmem + 128 * sb;        // S_j, then P_j
                wait(&s_full[sb], (gt / kTcSBufs) & 1);
                tc_fence_after_sync();
                float x[128];
                {
                    uint32_t v0[128];
#pragma unroll
                    for (int c = 0; c < kTcChunks; ++c)
                        tmem_ld32(tS + lane_addr + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(v0 + 32 * c));
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 128; ++e) x[e] = __uint_as_float(v0[e]);
                }
                // causal mask (only on tiles that reach past this row's
                // position) and the row max on the raw scores (the scale is
                // positive; eight independent partial maxima and sums keep
                // the dependency chains short)
                const int key0 = j * kTcKeys;
                float pm[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) pm[e] = -INFINITY;
                if (key0 + kTcKeys - 1 <= pos) {
#pragma unroll
                    for (int e = 0; e < 128; ++e) pm[e & 7] = fmaxf(pm[e & 7], x[e]);
                } else {
#pragma unroll
                    for (int e = 0; e < 128; ++e) {
                        x[e] = key0 + e <= pos ? x[e] : -INFINITY;
                        pm[e & 7] = fmaxf(pm[e & 7], x[e]);
                    }
                }
                const float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                                       fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7]))) * sl;   // log2 units
                // the reference max: raised only when the row max grows past 2^8
                const bool need = j > 0 && mx > m + kRescaleThresholdLog2;
                const float f = need ? ex2(m - mx) : 1.f;
                if (j == 0 || need) m = mx;                 // key 0 is visible to every row
                // P = 2^(x scale log2(e) - m), computed and stored into tensor
                // memory over S_j 32 keys at a time (the A operand of P V: keys
                // 2i, 2i+1 in column i of [0, 64), bf16 lo parts in [64, 128)),
                // before the previous product has finished; two keys per step
                // in packed fp32 (x sl - m, p - hi and the row sums each one
                // instruction for the pair)
                uint64_t ps[4];                              // partial sums, two lanes each
#pragma unroll
                for (int e = 0; e < 4; ++e) ps[e] = 0ull;
                const uint64_t sl2 = f32x2_pack(sl, sl), negm2 = f32x2_pack(-m, -m);
                const uint64_t minus1 = f32x2_pack(-1.f, -1.f);
#pragma unroll
                for (int c = 0; c < kTcChunks; ++c) {
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int e = 16 * c + i;
                        float a0, a1;
                        f32x2_unpack(f32x2_fma(f32x2_pack(x[2 * e], x[2 * e + 1]), sl2, negm2), a0, a1);
                        const float p0 = ex2(a0), p1 = ex2(a1);
                        if (kSplitP) {
                            // bf16 hi = p with its low 16 bits cut off (exact in
                            // fp32), lo = the remainder, also cut to bf16: hi +
                            // lo carries p to 2^-15, with integer and fp32 adds only
                            const float h0 = __uint_as_float(__float_as_uint(p0) & 0xffff0000u);
                            const float h1 = __uint_as_float(__float_as_uint(p1) & 0xffff0000u);
                            hi[i] = prmt(__float_as_uint(p0), __float_as_uint(p1), 0x7632u);
                            const uint64_t pp = f32x2_pack(p0, p1);
                            float d0, d1;
                            f32x2_unpack(f32x2_fma(f32x2_pack(h0, h1), minus1, pp), d0, d1);
                            lo[i] = prmt(__float_as_uint(d0), __float_as_uint(d1), 0x7632u);
                            ps[i & 3] = f32x2_add(ps[i & 3], pp);
                        } else {
                            hi[i] = M::pack(p0, p1);
                            const float2 u = M::unpack(hi[i]);
                            lo[i] = 0u;
                            ps[i & 3] = f32x2_add(ps[i & 3], f32x2_pack(u.x, u.y));
                        }
                    }
                    tmem_st16(tS + lane_addr + 16 * c, hi);
                    if (kSplitP) tmem_st16(tS + lane_addr + 64 + 16 * c, lo);
                }
                float q8[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) f32x2_unpack(ps[e], q8[2 * e], q8[2 * e + 1]);
                l = l * f + (((q8[0] + q8[1]) + (q8[2] + q8[3])) + ((q8[4] + q8[5]) + (q8[6] + q8[7])));
                // P_{j-1} V_{j-1} must be complete before O is rescaled
                const bool rescale = __any_sync(0xffffffffu, need);
                if (j > 0 && rescale) {
                    wait(&o_done[(gt - 1) % kTcSBufs], ((gt - 1) / kTcSBufs) & 1);
                    tc_fence_after_sync();
                }
                if (rescale) {
#pragma unroll
                    for (int c = 0; c < kTcChunks; ++c) {
                        uint32_t v[32];
                        tmem_ld32(tO + lane_addr + 32 * c, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * f);
                        tmem_st32(tO + lane_addr + 32 * c, v);
                    }
                }
                // the unit's last tile: V rows past the context may hold stale
                // bits; clear them
                if (key0 + kTcKeys > U.L) {
                    wait(&v_full[sv], (gt / kTcVStages) & 1);
                    if (key0 + r >= U.L) {
                        uint8_t* vd = smem + Lay::kV + sv * kTcOperand;
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            *reinterpret_cast<uint4*>(vd + tc_chunk(r, c)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                tmem_wait_st();
                fence_proxy_async_smem();                   // the cleared V rows
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[sb]);
            }
            // the next unit's Q into the other buffer now (its previous unit's
            // products have all completed: this unit's S products, issued
            // after them, have), so that its first products overlap this
            // unit's epilogue
            TcUnit N;
            bool next = false;
            for (; k < rounds && !next; ++k) next = unit_at(k, N);
            if (next) store_q(N, (nu + 1) & 1);
            // epilogue: O / l for the unit's rows, once its last product is
            // done; the next unit's first product overwrites O only after
            // this thread's P of that unit, which comes after these loads
            wait(&o_done[(gt - 1) % kTcSBufs], ((gt - 1) / kTcSBufs) & 1);
            tc_fence_after_sync();
            if (!failed) {
                const float inv = 1.f / l;
                T* out = reinterpret_cast<T*>(p.out) +
                         ((size_t)(U.q0 + U.t0 + min(t, U.rows - 1)) * p.num_q_heads + (size_t)U.g * G + h) * 128;
#pragma unroll
                for (int c = 0; c < kTcChunks; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tO + lane_addr + 32 * c, v);
                    tmem_wait_ld();
                    if (t < U.rows) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                w[e] = M::pack(__uint_as_float(v[8 * q + 2 * e]) * inv,
                                               __uint_as_float(v[8 * q + 2 * e + 1]) * inv);
                            *reinterpret_cast<uint4*>(out + 32 * c + 8 * q) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
            }
            U = N;
            have = next;
            ++nu;
        }
        if (failed && lane == 0) flag_error(p.err, PA_DEVERR_WAIT_TIMEOUT);
    }

    // every role is done with tensor memory
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTcCols);
    }
}

template <typename T>
cudaError_t launch_prefill_tc_t(const CUtensorMap& tmk, const CUtensorMap& tmv,
                                const PrefillParams& p, dim3 grid, cudaStream_t stream) {
    const int smem = TcLayout::kDynamicSmem;
    cudaError_t e = cudaFuncSetAttribute(paged_prefill_tc_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_with_pdl(paged_prefill_tc_kernel<T>, grid, dim3(kTcThreads), smem, stream, tmk,
                           tmv, p);
}

bool prefill_tc_supported(int head_dim, int group, float scale) {
    return head_dim == 128 && (group == 1 || group == 2 || group == 4 || group == 8) && scale > 0.f;
}

int prefill_tc_chunks(int group, int max_query_len) {
    const int qt = kTcRows / group;
    return (max_query_len + qt - 1) / qt;
}

// Counting sort of the items by key-tile count, descending; the order inside
// one count is whatever the atomics give (every item is computed alone, so
// the results do not depend on it).
constexpr int kPlanThreads = 1024;
constexpr int kPlanBuckets = 4096;               // counts above 4095 share the top bucket

__device__ __forceinline__ int prefill_item_tiles(const PrefillParams& p, int item) {
    const int b = item / p.max_chunks, qt = item % p.max_chunks, QT = kTcRows / p.group;
    const int max_ctx = p.max_blocks_per_seq * p.block_size;
    const int L = min(max(p.context_lens[b], 0), max_ctx);
    const int C = min(p.query_start[b + 1] - p.query_start[b], L);
    const int t0 = qt * QT;
    if (t0 >= C) return 0;
    return min((L - C + t0 + min(QT, C - t0) - 1) / kTcKeys + 1, kPlanBuckets - 1);
}

__global__ void __launch_bounds__(kPlanThreads, 1)
    prefill_tc_plan_kernel(const __grid_constant__ PrefillParams p, int32_t* sched) {
    __shared__ int offs[kPlanBuckets];
    __shared__ int warp_sum[kPlanThreads / 32];
    grid_dependency_wait();
    allow_dependent_launch();
    const int n = p.num_seqs * p.max_chunks, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    for (int c = tid; c < kPlanBuckets; c += kPlanThreads) offs[c] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kPlanThreads) atomicAdd(&offs[prefill_item_tiles(p, i)], 1);
    __syncthreads();
    // exclusive scan in descending count order: thread tid owns the four
    // buckets 4095 - 4 tid .. 4092 - 4 tid
    constexpr int kPer = kPlanBuckets / kPlanThreads;
    int own[kPer], sum = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        own[k] = offs[kPlanBuckets - 1 - (kPer * tid + k)];
        sum += own[k];
    }
    int incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
    }
    if (lane == 31) warp_sum[w] = incl;
    __syncthreads();
    if (w == 0) {
        int v = warp_sum[lane], vi = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, vi, d);
            if (lane >= d) vi += u;
        }
        warp_sum[lane] = vi - v;                       // exclusive over warps
    }
    __syncthreads();
    int run = warp_sum[w] + incl - sum;
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        offs[kPlanBuckets - 1 - (kPer * tid + k)] = run;
        run += own[k];
    }
    __syncthreads();
    for (int i = tid; i < n; i += kPlanThreads) {
        const int c = prefill_item_tiles(p, i);
        sched[atomicAdd(&offs[c], 1)] = c > 0 ? i : -1;
    }
}

cudaError_t launch_prefill_tc_plan(const PrefillParams& p, int32_t* sched, cudaStream_t stream) {
    return launch_with_pdl(prefill_tc_plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream, p, sched);
}

cudaError_t launch_prefill_tc(int dtype, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              const PrefillParams& p, int num_kv_heads, cudaStream_t stream) {
    // one persistent CTA per SM (shared and tensor memory hold one), each
    // walking its share of the units
    const int64_t units = (int64_t)p.num_seqs * p.max_chunks * num_kv_heads;
    if (units <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(units < sms ? units : sms));
    if (dtype == PA_BF16) return launch_prefill_tc_t<__nv_bfloat16>(tmk, tmv, p, grid, stream);
    return launch_prefill_tc_t<__half>(tmk, tmv, p, grid, stream);
}

}  // namespace pa
