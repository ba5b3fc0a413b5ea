// Chunked-prefill attention on the fifth-generation tensor cores (tcgen05,
// tensor-memory accumulators), head_dim 128 and GQA groups of 1, 2, 4 or 8.
//
// Sequence b holds L_b tokens, the last C_b of which are new; new token i
// sits at position L_b - C_b + i and attends causally to positions 0..itself
// (ta-paperlens page, prefill vs decode and the quadratic cost of prefill;
// techfeed summary, chunked prefill).  One CTA serves 128 query rows: 128 / G
// new tokens of one (sequence, KV head) times the G query heads that read
// that KV head, so every K/V tile is read once for all of them.
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
// softmax threads per query row: one (128 keys, four softmax warps, no row
// exchange) measured 4 % faster than two (64 keys each, eight warps, maxima
// and sums exchanged through shared memory), which was 3 % faster than four:
// fewer ALU-ready warps beside the MMA issuers on each scheduler
constexpr int kTcPerRow = 1;
constexpr int kTcRowKeys = 128 / kTcPerRow;   // keys (and output dims) of one thread
constexpr int kTcChunks = kTcRowKeys / 32;    // 32-column tensor-memory accesses of a thread
constexpr int kTcRowVec = kTcRowKeys / 8;     // 16-byte pieces of a thread's Q / V row slice
static_assert(kTcPerRow == 1 || kTcPerRow == 2 || kTcPerRow == 4, "1, 2 or 4 softmax threads per row");
constexpr int kTcSoftmaxWarps = 4 * kTcPerRow;

constexpr int kTcVWarp = 2 + kTcSoftmaxWarps;  // the V producer, after the softmax warps
constexpr int kTcPvWarp = 3 + kTcSoftmaxWarps; // issues P V (warp 1 issues S)
constexpr int kTcThreads = (4 + kTcSoftmaxWarps) * 32;
constexpr uint32_t kTcCols = 512;            // tensor-memory columns: S0/P0, S1/P1, S2/P2, O
constexpr int kTcOperand = 32768;            // 128 rows x 2 halves x 128 B
constexpr int kTcHalf = 16384;               // one 64-element half: 128 rows x 128 B

struct TcLayout {
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + kTcOperand;
    static constexpr int kV = kK + kTcKStages * kTcOperand;
    static constexpr int kBytes = kV + kTcVStages * kTcOperand;
    static constexpr int kDynamicSmem = kBytes + 1024;
    // with the ~6.2 KB of static shared memory (barriers, row exchange) this
    // must stay within the 227 KB a CTA may hold
    static_assert(kDynamicSmem + 6400 <= 232448, "shared memory over the per-CTA limit");
};

// Byte offset of 16-byte chunk c (elements 8c .. 8c+7 of 128) of row r in an
// operand of two 64-element halves with the 128-byte swizzle.
__device__ __forceinline__ int tc_chunk(int r, int c) {
    return (c >> 3) * kTcHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

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
    __shared__ float xchg[3][kTcPerRow][kTcRows];   // row maxima (two sets by tile parity), sums
    __shared__ __align__(8) uint64_t s_full[kTcSBufs], q_full, p_full[kTcSBufs], o_done[kTcSBufs];
    __shared__ uint32_t tmem_base;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.group;
    const int QT = kTcRows / G;                             // new tokens per CTA
    const int num_kv_heads = p.num_q_heads / G;

    grid_dependency_wait();
    allow_dependent_launch();
    // CTAs start in index order: rank r takes the r-th (sequence, chunk) item
    // of the schedule, for every KV head in turn
    const int g = (int)(blockIdx.x % (unsigned)num_kv_heads);
    const int rank = (int)(blockIdx.x / (unsigned)num_kv_heads);
    const int n_items = p.num_seqs * p.max_chunks;
    const int item = p.sched ? p.sched[rank] : n_items - 1 - rank;
    if (item < 0) return;
    const int b = item / p.max_chunks, qt = item % p.max_chunks;
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
    const int t0 = qt * QT;
    if (t0 >= C) return;
    const int rows = min(QT, C - t0);
    const int last_pos = L - C + t0 + rows - 1;             // the CTA's last query position
    const int n_tiles = last_pos / kTcKeys + 1;

    // producers' loads: K or V of tile j, 16-token boxes through the block
    // table; boxes wholly past the context are not loaded
    const int32_t* table = p.block_tables + (size_t)b * p.max_blocks_per_seq;
    // boxes of tile j: this lane's block id and token offset for box `lane`
    auto describe = [&](int j, int& nbox, int& blk, int& sub) {
        const int key0 = j * kTcKeys;
        nbox = min(8, (L - key0 + 15) / 16);
        blk = 0, sub = 0;
        if (lane < nbox) {
            const int tok = key0 + 16 * lane;
            blk = __ldg(table + tok / p.block_size);
            sub = tok % p.block_size;
        }
    };
    // one operand (K or V) of tile j into stage j % stages
    auto load = [&](const CUtensorMap* map, uint64_t* full, uint64_t* empty, int kind_off,
                    int stages, int j) -> bool {
        int nbox, blk, sub;
        describe(j, nbox, blk, sub);
        const int s = j % stages;
        bool ok = true;
        if (lane == 0) {
            if (j >= stages && !mbar_wait(&empty[s], ((j / stages) - 1) & 1)) {
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
        // registered by lane 0 above, earlier in this warp's program order):
        // two warp instructions per tile instead of sixteen single-lane ones
        uint8_t* dst = smem + kind_off + s * kTcOperand;
        if (lane < nbox) {
            tma_load_4d(dst + lane * kBox16Bytes, map, &full[s], 0, g, sub, blk);
            tma_load_4d(dst + kTcHalf + lane * kBox16Bytes, map, &full[s], kBoxElems, g, sub, blk);
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
        for (int i = 0; i < kTcSBufs; ++i) mbar_init(&s_full[i], 1);
        mbar_init(&q_full, kTcSoftmaxWarps);                // one arrival per softmax warp
        for (int i = 0; i < kTcSBufs; ++i) mbar_init(&p_full[i], kTcSoftmaxWarps);
        for (int i = 0; i < kTcSBufs; ++i) mbar_init(&o_done[i], 1);
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base, kTcCols);
    // Q row r = (token r / G, head r % G), rows past the chunk zero: each of
    // the row's softmax threads fetches its slice (dims kTcRowKeys part ..;
    // with one thread per row, the whole row)
    uint32_t qw[kTcRowKeys / 2];
    if (warp >= 2 && warp < kTcVWarp) {
        const int r = (warp & 3) * 32 + lane, part = (warp - 2) >> 2;
        const int t = r / G, h = r % G;
        const uint4* src = reinterpret_cast<const uint4*>(
            reinterpret_cast<const T*>(p.q) +
            ((size_t)(q0 + t0 + min(t, rows - 1)) * p.num_q_heads + (size_t)g * G + h) * 128);
#pragma unroll
        for (int c = 0; c < kTcRowVec; ++c) {
            const uint4 v = t < rows ? __ldg(src + kTcRowVec * part + c) : make_uint4(0u, 0u, 0u, 0u);
            qw[4 * c] = v.x, qw[4 * c + 1] = v.y, qw[4 * c + 2] = v.z, qw[4 * c + 3] = v.w;
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = tmem_base;
    const uint32_t tO = tmem + 128 * kTcSBufs;             // S_j / P_j in columns 128 (j % 3)

    if (warp == 0 || warp == kTcVWarp) {
        // ------------------------------------------------------------------
        // producers: K tiles (warp 0, free once S is computed, three stages)
        // and V tiles (warp 6, held until P V is done, two stages)
        // ------------------------------------------------------------------
        if (lane == 0) prefetch_tensor_map(warp == 0 ? &tmap_k : &tmap_v);
        // warp 0 streams K, warp 6 V, each at its own pace (issuing the
        // first K tiles before the CTA barrier measured 7 % slower: their
        // block-table reads hold the barrier up)
        bool ok = true;
        for (int j = 0; j < n_tiles && ok; ++j) {
            ok = warp == 0 ? load(&tmap_k, k_full, k_empty, Lay::kK, kTcKStages, j)
                           : load(&tmap_v, v_full, v_empty, Lay::kV, kTcVStages, j);
        }
    } else if (warp == 1 || warp == kTcPvWarp) {
        // ------------------------------------------------------------------
        // MMA issuers, one thread each on two schedulers: warp 1 issues S_j,
        // the last warp P_j V_j.  S_j overwrites P_{j-3}, so it waits for that
        // product (o_done of buffer j % 3); P V in order accumulates O.
        // ------------------------------------------------------------------
        if (lane == 0) {
            constexpr uint32_t kIdS = idesc_f16(kTcRows, kTcKeys, kBf16, false);
            constexpr uint32_t kIdPV = idesc_f16(kTcRows, 128, kBf16, true);
            bool ok = true;
            if (warp == 1) {
                ok = mbar_wait(&q_full, 0);
                tc_fence_after_sync();
                const uint32_t aQ = smem_u32(smem + Lay::kQ);
                for (int j = 0; j < n_tiles && ok; ++j) {
                    const int s = j % kTcKStages, sb = j % kTcSBufs;
                    ok = mbar_wait(&k_full[s], (j / kTcKStages) & 1);
                    if (ok && j >= kTcSBufs) ok = mbar_wait(&o_done[sb], (j / kTcSBufs - 1) & 1);
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
                    mma_commit(&k_empty[s]);                // S_j has read K_j
                }
            } else {
                for (int j = 0; j < n_tiles && ok; ++j) {
                    const int s = j % kTcVStages;
                    ok = mbar_wait(&p_full[j % kTcSBufs], (j / kTcSBufs) & 1);
                    if (ok) ok = mbar_wait(&v_full[s], (j / kTcVStages) & 1);
                    if (!ok) break;
                    tc_fence_after_sync();
                    const uint32_t aV = smem_u32(smem + Lay::kV + s * kTcOperand);
                    const uint32_t tP = tmem + 128 * (j % kTcSBufs);   // P_j over S_j
#pragma unroll
                    for (int part = 0; part < (kSplitP ? 2 : 1); ++part) {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_f16_ts(tO, tP + 64 * part + 8 * kk,
                                       smem_desc_sw128(aV + kk * 16 * 128, kTcHalf, 1024), kIdPV,
                                       j > 0 || part > 0 || kk > 0);
                    }
                    mma_commit(&o_done[j % kTcSBufs]);
                    mma_commit(&v_empty[s]);                // P_j V_j has read V_j
                }
            }
            if (!ok) flag_error(p.err, PA_DEVERR_WAIT_TIMEOUT);
        }
    } else {
        // ------------------------------------------------------------------
        // softmax and epilogue: this thread owns slice `part` (kTcRowKeys keys
        // of each tile, kTcRowKeys output dims) of row r (tensor-memory lane
        // r); with more than one thread per row they exchange maxima and sums
        // through shared memory
        // ------------------------------------------------------------------
        const int r = (warp & 3) * 32 + lane, part = (warp - 2) >> 2;
        const int t = r / G, h = r % G;
        const int pos = min(L - C + t0 + t, L - 1);
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t my_cols = lane_addr + kTcRowKeys * part;
        const float sl = p.scale_log2;
        float m = -INFINITY, l = 0.f;
        // this thread's slice of its Q row into shared memory, laid out like
        // a K tile (the A operand of S); visible to the tensor cores after the
        // proxy fence
#pragma unroll
        for (int c = 0; c < kTcRowVec; ++c)
            *reinterpret_cast<uint4*>(smem + Lay::kQ + tc_chunk(r, kTcRowVec * part + c)) =
                make_uint4(qw[4 * c], qw[4 * c + 1], qw[4 * c + 2], qw[4 * c + 3]);
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_full);
        bool failed = false;                 // a wait ran out: finish the loop without waiting
        auto wait = [&](uint64_t* bar, uint32_t parity) {
            if (!failed && !__all_sync(0xffffffffu, mbar_wait(bar, parity))) failed = true;
        };
        // the row's threads' values, through shared set `set`
        auto exchange = [&](int set, float v) {
            if (kTcPerRow == 1) return make_float4(v, 0.f, 0.f, 0.f);
            xchg[set][part][r] = v;
            // the row's threads sit in the softmax warps of lane quarter
            // warp % 4: one named barrier (1 + warp % 4) per quarter
            asm volatile("bar.sync %0, %1;" ::"r"(1 + (warp & 3)), "n"(kTcPerRow * 32) : "memory");
            if (kTcPerRow == 2) return make_float4(xchg[set][0][r], xchg[set][1][r], 0.f, 0.f);
            return make_float4(xchg[set][0][r], xchg[set][1][r], xchg[set][2][r], xchg[set][3][r]);
        };
        for (int j = 0; j < n_tiles; ++j) {
            const int bb = j & 1, s = j % kTcVStages, sb = j % kTcSBufs;
            const uint32_t tS = tmem + 128 * sb;            // S_j, then P_j
            wait(&s_full[sb], (j / kTcSBufs) & 1);
            tc_fence_after_sync();
            float x[kTcRowKeys];
            {
                uint32_t v0[kTcRowKeys];
#pragma unroll
                for (int c = 0; c < kTcChunks; ++c)
                    tmem_ld32(tS + my_cols + 32 * c,
                              *reinterpret_cast<uint32_t(*)[32]>(v0 + 32 * c));
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < kTcRowKeys; ++k) x[k] = __uint_as_float(v0[k]);
            }
            // causal mask (only on tiles that reach past this row's position)
            // and the row max over the row's threads, on the raw scores (the
            // scale is positive; eight independent partial maxima and sums
            // keep the dependency chains short)
            const int key0 = j * kTcKeys + kTcRowKeys * part;
            float pm[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) pm[e] = -INFINITY;
            if (key0 + kTcRowKeys - 1 <= pos) {
#pragma unroll
                for (int k = 0; k < kTcRowKeys; ++k) pm[k & 7] = fmaxf(pm[k & 7], x[k]);
            } else {
#pragma unroll
                for (int k = 0; k < kTcRowKeys; ++k) {
                    x[k] = key0 + k <= pos ? x[k] : -INFINITY;
                    pm[k & 7] = fmaxf(pm[k & 7], x[k]);
                }
            }
            float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                             fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
            {
                // two column sets by tile parity: a set is rewritten only after
                // every thread has passed the next tile's barrier
                const float4 e4 = exchange(bb, mx);
                mx = (kTcPerRow == 1   ? e4.x
                      : kTcPerRow == 2 ? fmaxf(e4.x, e4.y)
                                       : fmaxf(fmaxf(e4.x, e4.y), fmaxf(e4.z, e4.w))) * sl;   // log2 units
            }
            // the reference max: raised only when the row max grows past 2^8
            const bool need = j > 0 && mx > m + kRescaleThresholdLog2;
            const float f = need ? ex2(m - mx) : 1.f;
            if (j == 0 || need) m = mx;                     // key 0 is visible to every row
            // P = 2^(x scale log2(e) - m), computed and stored into tensor
            // memory over S_j one 32-key chunk at a time (the A operand of P V:
            // keys 2i, 2i+1 in column i of [0, 64), bf16 lo parts in [64, 128);
            // this thread's 64 keys are 32 columns at 32 part), before the
            // previous product has finished; two keys per step in packed fp32
            // (x sl - m, p - hi and the row sums each one instruction for the pair)
            uint64_t ps[4];                                  // partial sums, two lanes each
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
                        // bf16 hi = p with its low 16 bits cut off (exact in fp32),
                        // lo = the remainder, also cut to bf16: hi + lo carries p to
                        // 2^-15, with integer and fp32 adds only
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
                const uint32_t col = lane_addr + (kTcRowKeys / 2) * part + 16 * c;
                tmem_st16(tS + col, hi);
                if (kSplitP) tmem_st16(tS + 64 + col, lo);
            }
            float q8[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) f32x2_unpack(ps[e], q8[2 * e], q8[2 * e + 1]);
            l = l * f + (((q8[0] + q8[1]) + (q8[2] + q8[3])) + ((q8[4] + q8[5]) + (q8[6] + q8[7])));
            // P_{j-1} V_{j-1} must be complete before O is rescaled
            const bool rescale = __any_sync(0xffffffffu, need);
            if (j > 0 && rescale) {
                wait(&o_done[(j - 1) % kTcSBufs], ((j - 1) / kTcSBufs) & 1);
                tc_fence_after_sync();
            }
            if (rescale) {
#pragma unroll
                for (int c = 0; c < kTcChunks; ++c) {
                    uint32_t v[32];
                    tmem_ld32(tO + my_cols + 32 * c, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * f);
                    tmem_st32(tO + my_cols + 32 * c, v);
                }
                tmem_wait_st();
            }
            // the last tile: V rows past the context may hold stale bits; clear them
            if (j * kTcKeys + kTcKeys > L) {
                wait(&v_full[s], (j / kTcVStages) & 1);
                if (j * kTcKeys + r >= L) {
                    uint8_t* vd = smem + Lay::kV + s * kTcOperand;
#pragma unroll
                    for (int c = kTcRowVec * part; c < kTcRowVec * (part + 1); ++c)
                        *reinterpret_cast<uint4*>(vd + tc_chunk(r, c)) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            tmem_wait_st();
            fence_proxy_async_smem();                       // the cleared V rows
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[sb]);
        }
        // epilogue: O / l for the chunk's rows, l summed over the row's threads
        wait(&o_done[(n_tiles - 1) % kTcSBufs], ((n_tiles - 1) / kTcSBufs) & 1);
        tc_fence_after_sync();
        const float4 l4 = exchange(2, l);
        if (!failed) {
            const float inv = 1.f / (kTcPerRow == 1   ? l4.x
                                     : kTcPerRow == 2 ? l4.x + l4.y
                                                      : (l4.x + l4.y) + (l4.z + l4.w));
            T* out = reinterpret_cast<T*>(p.out) +
                     ((size_t)(q0 + t0 + min(t, rows - 1)) * p.num_q_heads + (size_t)g * G + h) * 128 +
                     kTcRowKeys * part;
#pragma unroll
            for (int c = 0; c < kTcChunks; ++c) {
                uint32_t v[32];
                tmem_ld32(tO + my_cols + 32 * c, v);
                tmem_wait_ld();
                if (t < rows) {
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
        } else if (lane == 0) {
            flag_error(p.err, PA_DEVERR_WAIT_TIMEOUT);
        }
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
    dim3 grid((unsigned)((int64_t)p.num_seqs * p.max_chunks * num_kv_heads));
    if (dtype == PA_BF16) return launch_prefill_tc_t<__nv_bfloat16>(tmk, tmv, p, grid, stream);
    return launch_prefill_tc_t<__half>(tmk, tmv, p, grid, stream);
}

}  // namespace pa
