// Per-warp attention over one 16-token tile of one (sequence, KV head), the
// building block of every decode kernel.
//
// A 16-bit tile in shared memory is D/64 boxes of [16 tokens][128 B] (2 KiB
// each) with the 128-byte swizzle TMA writes: 16-byte chunk c of row r sits
// at chunk c ^ (r % 8).  Fragment roles (m16n8k16, r8 = lane/4, c4 = lane%4):
//   S^T[t][h] = K[t][:] . q[h][:]        A = K tile (16 tokens x 16 dims),
//                                        B = q^T (16 dims x 8 heads)
//   O^T[d][h] += V^T[d][:] . P^T[:][h]   A = V^T (16 dims x 16 tokens),
//                                        B = P^T (16 tokens x 8 heads)
// so a lane holds scores of tokens r8 and r8+8 for heads 2c4, 2c4+1, and
// accumulators of dims r8, r8+8 (per 16-dim slab) for the same two heads.
// The G <= 8 query heads of the group are the 8 columns; columns >= G are
// zero.  Online softmax in log2 units with a lazily raised running max (the
// accumulator is rescaled only when a tile's max exceeds the max in use by
// more than 2^8; numerator and denominator share the reference max, so the
// result is exact in real arithmetic).  P is rounded to the 16-bit type --
// for bf16 as a hi + lo pair (~2^-17 together) -- and transposed in
// registers with movmatrix.
#pragma once

#include <type_traits>

#include "pa_device.cuh"

namespace pa {

constexpr int kBox16Bytes = kTileTokens * 128;       // one [16][128 B] box
constexpr float kRescaleThresholdLog2 = 8.0f;        // rescale when the max grows > 2^8

template <int D>
struct TileState {
    float acc[D / 16][4];     // O^T slabs of 16 dims
    float mA, mB;             // reference max in use (log2 units)
    float tA, tB;             // true running max (log2 units)
    float lA, lB;             // this lane's share of the row sums

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int n = 0; n < D / 16; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        mA = mB = tA = tB = -INFINITY;
        lA = lB = 0.f;
    }

    // Row sums across the 8 lanes that share a head pair.
    __device__ __forceinline__ void reduce_row_sums() {
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            lA += __shfl_xor_sync(0xffffffffu, lA, o);
            lB += __shfl_xor_sync(0xffffffffu, lB, o);
        }
    }
};

// q^T as the B operand: b0 = q[r8][16kk + 2c4 ..], b1 = q[r8][16kk + 8 + 2c4 ..];
// rows >= G are zero.  q_group points at the group's first query head.
template <typename T, int D>
__device__ __forceinline__ void load_q_fragments(uint32_t (&qb)[D / 16][2], const T* q_group,
                                                 int G, int lane) {
    const int r8 = lane >> 2, c4 = lane & 3;
    const bool valid = r8 < G;
    const T* qrow = q_group + (valid ? r8 : 0) * D;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        qb[kk][0] = valid ? __ldg(reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 2 * c4)) : 0u;
        qb[kk][1] = valid ? __ldg(reinterpret_cast<const uint32_t*>(qrow + kk * 16 + 8 + 2 * c4)) : 0u;
    }
}

// ---------------------------------------------------------------------------
// FP8 (E4M3) tiles, D = 128: the staged tile is one box of [16 tokens][128 B]
// codes per K and per V (128 B swizzle), and the products run in fp16 straight
// from registers.  E4M3 codes are exact in fp16, so the staged values enter the
// tensor cores unchanged; q is brought to fp16 once per warp (see
// load_q_fragments_fp8) and P is rounded to fp16 once.
//
// The contraction and output orders are permuted so that every lane reads
// whole 16-byte chunks:
//   S^T = K q^T: in k-step kk, lane (r8, c4)'s four k positions (2c4, 2c4+1,
//     2c4+8, 2c4+9) stand for dims 32 c4 + 4 kk + (0, 1, 2, 3): the lane reads
//     bytes [32 c4, 32 c4 + 32) of token rows r8 and r8 + 8, and q is loaded
//     with the same order.
//   O^T += V^T P^T: slab n's rows r8 and r8 + 8 stand for dims 16 r8 + 2n and
//     16 r8 + 2n + 1, so the lane reads bytes [16 r8, 16 r8 + 16) of token rows
//     2c4, 2c4+1, 2c4+8, 2c4+9 and pairs bytes of two tokens with prmt.
// Accumulator slab n of a lane therefore holds dims 16 r8 + 2n (c0, c1) and
// 16 r8 + 2n + 1 (c2, c3); fp8_dims() gives them to the epilogues.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void fp8_dims(int n, int r8, int& d_lo, int& d_hi) {
    d_lo = 16 * r8 + 2 * n;
    d_hi = d_lo + 1;
}

// 16-byte shared-memory load.  The tile pointers come from an aligned
// integer offset of the dynamic shared buffer, so a plain dereference would
// compile to a generic load; this one is a shared load.
__device__ __forceinline__ uint4 lds128(const uint8_t* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

// 8-byte shared-memory load (shared-window address).
__device__ __forceinline__ void lds64(uint32_t addr, uint32_t& a, uint32_t& b) {
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "r"(addr));
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int j) {
    return j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// q of the group as fp16 B fragments in the FP8 dim order, scaled by 2^-s so
// that fp16 holds it; returns s.  An fp16 q is taken as it is (s = 0); a bf16
// q is scaled so that the group's largest magnitude lands in [2^14, 2^15),
// which keeps every value within fp16's range and its 11 significant bits
// for all but values 2^-24 below the largest.  Rows >= G are zero.
template <typename T>
__device__ __forceinline__ int load_q_fragments_fp8(uint32_t (&qb)[8][2], const T* q_group, int G,
                                                    int lane) {
    const int r8 = lane >> 2, c4 = lane & 3;
    const bool valid = r8 < G;
    const uint4* src = reinterpret_cast<const uint4*>(q_group + (valid ? r8 : 0) * 128 + 32 * c4);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = valid ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
        w[4 * i] = v.x, w[4 * i + 1] = v.y, w[4 * i + 2] = v.z, w[4 * i + 3] = v.w;
    }
    if constexpr (std::is_same<T, __half>::value) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) qb[kk][0] = w[2 * kk], qb[kk][1] = w[2 * kk + 1];
        return 0;
    } else {
        float mx = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float2 f = Mma<T>::unpack(w[i]);
            mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        int e = 0;
        (void)frexpf(mx, &e);                        // mx < 2^e (e = 0 for mx = 0)
        const int s = min(100, max(-100, e - 15));
        const float f = __int_as_float((127 - s) << 23);   // 2^-s, exact
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const float2 v = Mma<T>::unpack(w[2 * kk + j]);
                qb[kk][j] = Mma<__half>::pack(v.x * f, v.y * f);
            }
        }
        return s;
    }
}

// Writes 8 codes (8 dims, chunk c of 16) into token row r of an FP8 tile.
__device__ __forceinline__ void put_code_chunk(uint8_t* tile, int r, int c, uint2 codes) {
    *reinterpret_cast<uint2*>(tile + r * 128 + (((c >> 1) ^ (r & 7)) << 4) + (c & 1) * 8) = codes;
}

// Pieces of the FP8 tile math.  K: lane (r8, c4) reads 16-byte chunks
// 2c4, 2c4+1 of token rows r8 and r8 + 8 (same swizzle row phase); k-step kk
// takes word kk & 3 of chunk kk >> 2.  V: chunk r8 of token rows 2c4, 2c4+1,
// 2c4+8, 2c4+9, cleared for rows past the end (they may hold stale codes,
// NaN among them).
__device__ __forceinline__ void fp8_load_k(uint4 (&klo)[2], uint4 (&khi)[2], const uint8_t* ktile,
                                           int lane) {
    const int r8 = lane >> 2, c4 = lane & 3;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int off = (((2 * c4 + i) ^ r8) << 4);
        klo[i] = lds128(ktile + r8 * 128 + off);
        khi[i] = lds128(ktile + (r8 + 8) * 128 + off);
    }
}

__device__ __forceinline__ void fp8_score_step(float (&sc)[4], const uint4 (&klo)[2],
                                               const uint4 (&khi)[2], int kk, uint32_t b0,
                                               uint32_t b1) {
    uint32_t a0, a1, a2, a3;
    e4m3x4_to_f16x2x2(word_of(klo[kk >> 2], kk & 3), a0, a2);
    e4m3x4_to_f16x2x2(word_of(khi[kk >> 2], kk & 3), a1, a3);
    Mma<__half>::run(sc, a0, a1, a2, a3, b0, b1);
}

__device__ __forceinline__ void fp8_load_v(uint4 (&v)[4], const uint8_t* vtile, int tok0,
                                           int t_end, int lane) {
    const int r8 = lane >> 2, c4 = lane & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = 2 * c4 + (i & 1) + 8 * (i >> 1);
        v[i] = lds128(vtile + t * 128 + ((r8 ^ (t & 7)) << 4));
    }
    if (tok0 + kTileTokens > t_end) {               // ragged tail only (warp-uniform)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (tok0 + 2 * c4 + (i & 1) + 8 * (i >> 1) >= t_end) v[i] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// O^T slab n += V^T . P^T from the staged codes (two tokens' bytes paired by prmt).
__device__ __forceinline__ void fp8_pv_slab(float (&acc)[4], const uint4 (&v)[4], int n,
                                            uint32_t pb0, uint32_t pb1) {
    const int j = n >> 1;
    const uint32_t sel = (n & 1) ? 0x7362u : 0x5140u;   // bytes (2h, 2h+1) of two tokens
    const uint32_t x01 = prmt(word_of(v[0], j), word_of(v[1], j), sel);
    const uint32_t x23 = prmt(word_of(v[2], j), word_of(v[3], j), sel);
    uint32_t a0, a1, a2, a3;
    e4m3x4_to_f16x2x2(x01, a0, a1);
    e4m3x4_to_f16x2x2(x23, a2, a3);
    Mma<__half>::run(acc, a0, a1, a2, a3, pb0, pb1);
}

// Raises the reference maxima when this step's maxima xa, xb (log2 units, per
// head pair, already reduced over the warp) exceed them by more than 2^8.
__device__ __forceinline__ void fp8_raise(TileState<128>& s, float xa, float xb) {
    s.tA = fmaxf(s.tA, xa);
    s.tB = fmaxf(s.tB, xb);
    const bool raiseA = xa > s.mA + kRescaleThresholdLog2;
    const bool raiseB = xb > s.mB + kRescaleThresholdLog2;
    if (__any_sync(0xffffffffu, raiseA || raiseB)) {
        const float nA = raiseA ? xa : s.mA, nB = raiseB ? xb : s.mB;
        const float fA = ex2(s.mA - nA), fB = ex2(s.mB - nB);
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            s.acc[n][0] *= fA;
            s.acc[n][1] *= fB;
            s.acc[n][2] *= fA;
            s.acc[n][3] *= fB;
        }
        s.lA *= fA;
        s.lB *= fB;
        s.mA = nA;
        s.mB = nB;
    }
}

// Masked, scaled scores (r8 / r8 + 8 rows, heads hA / hB) of a tile at tok0.
__device__ __forceinline__ void fp8_mask(float (&x)[4], const float (&sc)[4], int tok0, int t_end,
                                         float scale_log2, int lane) {
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = sc[i] * scale_log2;
    if (tok0 + kTileTokens > t_end) {               // ragged tail only (warp-uniform)
        const int r8 = lane >> 2;
        if (tok0 + r8 >= t_end) x[0] = x[1] = -INFINITY;
        if (tok0 + r8 + 8 >= t_end) x[2] = x[3] = -INFINITY;
    }
}

// P of a tile in fp16 (added into the row sums), transposed into P^T fragments.
__device__ __forceinline__ void fp8_probs(TileState<128>& s, const float (&x)[4], uint32_t& pb0,
                                          uint32_t& pb1) {
    using M = Mma<__half>;
    const uint32_t p01 = M::pack(ex2(x[0] - s.mA), ex2(x[1] - s.mB));
    const uint32_t p23 = M::pack(ex2(x[2] - s.mA), ex2(x[3] - s.mB));
    const float2 u = M::unpack(p01), w = M::unpack(p23);
    s.lA += u.x + w.x;
    s.lB += u.y + w.y;
    pb0 = movmatrix_trans(p01);
    pb1 = movmatrix_trans(p23);
}

__device__ __forceinline__ void warp_max_pairs(float& xa, float& xb) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, o));
        xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, o));
    }
}

// Attends one FP8 tile (tokens tok0 .. tok0+15, masked from t_end on);
// qfrag(kk, b0, b1) supplies the fp16 q^T fragments of k-step kk.
// release() runs once the warp has read the staged codes into registers, so
// the stage can be refilled while the P V products run.
template <typename QFrag, typename Release>
__device__ __forceinline__ void attend_tile_fp8(TileState<128>& s, QFrag&& qfrag,
                                                const uint8_t* ktile, const uint8_t* vtile,
                                                int tok0, int t_end, float scale_log2, int lane,
                                                Release&& release) {
    uint4 klo[2], khi[2];
    fp8_load_k(klo, khi, ktile, lane);
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        uint32_t b0, b1;
        qfrag(kk, b0, b1);
        fp8_score_step(sc, klo, khi, kk, b0, b1);
    }
    uint4 v[4];
    fp8_load_v(v, vtile, tok0, t_end, lane);
    release();

    float x[4];
    fp8_mask(x, sc, tok0, t_end, scale_log2, lane);
    float xa = fmaxf(x[0], x[2]), xb = fmaxf(x[1], x[3]);
    warp_max_pairs(xa, xb);
    fp8_raise(s, xa, xb);
    uint32_t pb0, pb1;
    fp8_probs(s, x, pb0, pb1);
#pragma unroll
    for (int n = 0; n < 8; ++n) fp8_pv_slab(s.acc[n], v, n, pb0, pb1);
}

// Attends two FP8 tiles at once: tile 0 (tokens tok0 .. tok0+15) and tile 1
// (the next 16), both masked from t_end on.  Their score chains interleave,
// one max reduction and one rescale test cover both, and each accumulator
// slab takes both P V products, so the per-tile chain of dependent steps is
// about halved.  release() runs once both tiles' codes are in registers.
template <typename QFrag, typename Release>
__device__ __forceinline__ void attend_pair_fp8(TileState<128>& s, QFrag&& qfrag,
                                                const uint8_t* ktile0, const uint8_t* vtile0,
                                                const uint8_t* ktile1, const uint8_t* vtile1,
                                                int tok0, int t_end, float scale_log2, int lane,
                                                Release&& release) {
    uint4 klo0[2], khi0[2], klo1[2], khi1[2];
    fp8_load_k(klo0, khi0, ktile0, lane);
    fp8_load_k(klo1, khi1, ktile1, lane);
    float sc0[4] = {0.f, 0.f, 0.f, 0.f}, sc1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        uint32_t b0, b1;
        qfrag(kk, b0, b1);
        fp8_score_step(sc0, klo0, khi0, kk, b0, b1);
        fp8_score_step(sc1, klo1, khi1, kk, b0, b1);
    }
    uint4 v0[4], v1[4];
    fp8_load_v(v0, vtile0, tok0, t_end, lane);
    fp8_load_v(v1, vtile1, tok0 + kTileTokens, t_end, lane);
    release();

    float x[4], y[4];
    fp8_mask(x, sc0, tok0, t_end, scale_log2, lane);
    fp8_mask(y, sc1, tok0 + kTileTokens, t_end, scale_log2, lane);
    float xa = fmaxf(fmaxf(x[0], x[2]), fmaxf(y[0], y[2]));
    float xb = fmaxf(fmaxf(x[1], x[3]), fmaxf(y[1], y[3]));
    warp_max_pairs(xa, xb);
    fp8_raise(s, xa, xb);
    uint32_t pb0, pb1, qb0, qb1;
    fp8_probs(s, x, pb0, pb1);
    fp8_probs(s, y, qb0, qb1);
#pragma unroll
    for (int n = 0; n < 8; ++n) {
        fp8_pv_slab(s.acc[n], v0, n, pb0, pb1);
        fp8_pv_slab(s.acc[n], v1, n, qb0, qb1);
    }
}

// Writes one 16-byte chunk (8 dims) into row r of a 16-bit tile.
__device__ __forceinline__ void put_tile_chunk(uint8_t* tile, int r, int c, uint4 val) {
    *reinterpret_cast<uint4*>(tile + (c >> 3) * kBox16Bytes + r * 128 + (((c & 7) ^ (r & 7)) << 4)) =
        val;
}

// qfrag(kk, b0, b1) supplies the q^T B-operand fragments of k-step kk (from
// registers or from shared memory, as the caller keeps them).
// Attends the 16 tokens tok0 .. tok0+15 of a tile; tokens >= t_end are masked
// (their V rows are zeroed in shared memory, since they may hold stale
// non-finite bits).
template <typename T, int D, typename QFrag>
__device__ __forceinline__ void attend_tile(TileState<D>& s, QFrag&& qfrag,
                                            uint8_t* ktile, uint8_t* vtile, int tok0, int t_end,
                                            float scale_log2, int lane) {
    using M = Mma<T>;
    constexpr int kKSteps = D / 16;
    constexpr bool kSplitP = std::is_same<T, __nv_bfloat16>::value;
    const int r8 = lane >> 2;
    // ldmatrix row addresses: matrix j = lane/8 supplies row lane%8.
    // K (A operand, no transpose): j -> (tokens 8*(j&1).., dims hi = j>>1)
    const int k_tok = ((lane >> 3) & 1) * 8 + (lane & 7);
    const int k_hi = lane >> 4;
    // V (A operand of V^T, transposed): j -> (tokens 8*(j>>1).., dims hi = j&1)
    const int v_tok = (lane >> 4) * 8 + (lane & 7);
    const int v_hi = (lane >> 3) & 1;
    const uint32_t kbase = smem_u32(ktile);
    const uint32_t vbase = smem_u32(vtile);

    // S^T for the 16 tokens of the tile
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < kKSteps; ++kk) {
        const int chunk = 2 * kk + k_hi;                     // 16-byte chunk along D
        const uint32_t addr = kbase + (chunk >> 3) * kBox16Bytes + k_tok * 128 +
                              (((chunk & 7) ^ (k_tok & 7)) << 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(addr, a0, a1, a2, a3);
        uint32_t b0, b1;
        qfrag(kk, b0, b1);
        M::run(sc, a0, a1, a2, a3, b0, b1);
    }

    // mask past the span's end, scale into log2 units
    const bool v_lo = tok0 + r8 < t_end, v_hi8 = tok0 + r8 + 8 < t_end;
    const float x0 = v_lo ? sc[0] * scale_log2 : -INFINITY;    // (r8,   hA)
    const float x1 = v_lo ? sc[1] * scale_log2 : -INFINITY;    // (r8,   hB)
    const float x2 = v_hi8 ? sc[2] * scale_log2 : -INFINITY;   // (r8+8, hA)
    const float x3 = v_hi8 ? sc[3] * scale_log2 : -INFINITY;   // (r8+8, hB)
    float xa = fmaxf(x0, x2), xb = fmaxf(x1, x3);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, o));
        xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, o));
    }
    s.tA = fmaxf(s.tA, xa);
    s.tB = fmaxf(s.tB, xb);
    const bool raiseA = xa > s.mA + kRescaleThresholdLog2;
    const bool raiseB = xb > s.mB + kRescaleThresholdLog2;
    if (__any_sync(0xffffffffu, raiseA || raiseB)) {
        const float nA = raiseA ? xa : s.mA, nB = raiseB ? xb : s.mB;
        const float fA = ex2(s.mA - nA), fB = ex2(s.mB - nB);
#pragma unroll
        for (int n = 0; n < kKSteps; ++n) {
            s.acc[n][0] *= fA;
            s.acc[n][1] *= fB;
            s.acc[n][2] *= fA;
            s.acc[n][3] *= fB;
        }
        s.lA *= fA;
        s.lB *= fB;
        s.mA = nA;
        s.mB = nB;
    }
    // P in the 16-bit type; P^T fragments by an in-register transpose
    const float e0 = ex2(x0 - s.mA), e1 = ex2(x1 - s.mB);   // token r8
    const float e2 = ex2(x2 - s.mA), e3 = ex2(x3 - s.mB);   // token r8+8
    const uint32_t p01 = M::pack(e0, e1);
    const uint32_t p23 = M::pack(e2, e3);
    const uint32_t pb0 = movmatrix_trans(p01);   // (head r8, tokens 2c4..+1)
    const uint32_t pb1 = movmatrix_trans(p23);   // (head r8, tokens 8+2c4..+1)
    uint32_t pl0 = 0u, pl1 = 0u;
    if (kSplitP) {
        const float2 u = M::unpack(p01), w = M::unpack(p23);
        pl0 = movmatrix_trans(M::pack(e0 - u.x, e1 - u.y));
        pl1 = movmatrix_trans(M::pack(e2 - w.x, e3 - w.y));
        s.lA += e0 + e2;
        s.lB += e1 + e3;
    } else {
        const float2 u = M::unpack(p01), w = M::unpack(p23);
        s.lA += u.x + w.x;
        s.lB += u.y + w.y;
    }

    // ragged tail: zero V rows past the end so that 0 * V stays 0
    if (tok0 + kTileTokens > t_end) {
        const int valid = t_end - tok0;
        const int rows = kTileTokens - valid;
        for (int idx = lane; idx < (D / 64) * rows * 8; idx += 32) {
            const int hh = idx / (rows * 8);
            const int rem = idx - hh * rows * 8;
            const int rr = valid + (rem >> 3);
            *reinterpret_cast<uint4*>(vtile + hh * kBox16Bytes + rr * 128 + ((rem & 7) << 4)) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
    }

    // O^T += V^T . P^T, one m16n8k16 per 16-dim slab
#pragma unroll
    for (int n = 0; n < kKSteps; ++n) {
        const int chunk = 2 * n + v_hi;
        const uint32_t addr = vbase + (chunk >> 3) * kBox16Bytes + v_tok * 128 +
                              (((chunk & 7) ^ (v_tok & 7)) << 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(addr, a0, a1, a2, a3);
        M::run(s.acc[n], a0, a1, a2, a3, pb0, pb1);
        if (kSplitP) M::run(s.acc[n], a0, a1, a2, a3, pl0, pl1);
    }
}

}  // namespace pa
