// Internal declarations shared by the C-ABI layer and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

constexpr int kTileTokens = 16;      // tokens per pipeline tile (one box row count)
constexpr int kBoxElems = 64;        // innermost box extent: 64 x 2 B = one 128 B swizzle row
#ifndef PA_DECODE_CONSUMER_WARPS
#define PA_DECODE_CONSUMER_WARPS 2
#endif
constexpr int kConsumerWarps = PA_DECODE_CONSUMER_WARPS;  // warps that compute; +1 issues TMA
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
#ifndef PA_DECODE_STAGES
#define PA_DECODE_STAGES 4
#endif
#ifndef PA_DECODE_MIN_CTAS_PER_SM
#define PA_DECODE_MIN_CTAS_PER_SM 6
#endif
constexpr int kStages = PA_DECODE_STAGES;   // tiles in flight per CTA
constexpr int kMinCtasPerSm = PA_DECODE_MIN_CTAS_PER_SM;
// Consumer warp w takes tiles w, w + W, w + 2W, ... and tile i sits in stage
// i % kStages.  With kStages a multiple of W every stage belongs to exactly
// one warp, which waits on its phases in order; otherwise two warps would
// share a stage and a parity wait could match a phase two laps old.
static_assert(kStages % kConsumerWarps == 0, "stages must be a multiple of consumer warps");
// The FP8 cache halves the bytes of a tile, so its ring is twice as deep;
// its warps build fragments from the staged codes in registers, and six
// CTAs per SM (96 registers a thread) beat four or five on long contexts.
#ifndef PA_DECODE_MIN_CTAS_PER_SM_FP8
#define PA_DECODE_MIN_CTAS_PER_SM_FP8 6
#endif
#ifndef PA_DECODE_STAGES_FP8
#define PA_DECODE_STAGES_FP8 (2 * PA_DECODE_STAGES)
#endif
constexpr int kStagesFp8 = PA_DECODE_STAGES_FP8;
constexpr int kMinCtasPerSmFp8 = PA_DECODE_MIN_CTAS_PER_SM_FP8;
static_assert(kStagesFp8 % kConsumerWarps == 0, "stages must be a multiple of consumer warps");
// Tiles the decode producer issues per round (one lane per TMA box); two
// measured best: four delays the first copies of a round behind the last
// stage it waits for (shared-prefix batch 148 against 132 us).
#ifndef PA_DECODE_ISSUE_BATCH
#define PA_DECODE_ISSUE_BATCH 2
#endif
constexpr int kIssueBatch = PA_DECODE_ISSUE_BATCH;
// A wait on a pipeline barrier gives up after this many nanoseconds and
// reports PA_DEVERR_WAIT_TIMEOUT instead of spinning forever.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kMaxGroup = 8;         // query heads per KV head served by one CTA
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct DecodeParams {
    const void* q;                 // [B][Hq][D]
    const int32_t* block_tables;   // [B][MB]
    const int32_t* context_lens;   // [B]
    void* out;                     // [B][Hq][D] (single pass)
    float* tmp_out;                // [B][Hq][S][D] (split)
    float* max_logits;             // [B][Hq][S]
    float* exp_sums;               // [B][Hq][S]
    int* err;                      // device error word
    float scale_log2;              // scale * log2(e)
    int num_q_heads;
    int group;                     // Hq / Hkv
    int max_blocks_per_seq;
    int block_size;
    int64_t num_blocks;
    int partition_tokens;          // split: partition size; single pass: 0
    int max_parts;                 // split: S
    // fused layer-step only
    const void* k_new;             // [B][Hkv][D] new token of each sequence
    const void* v_new;
    const int64_t* slot_mapping;   // [B] slot of position L_b - 1 (negative: none)
    void* k_cache;                 // written at the new token's slot
    void* v_cache;
    int* counters;                 // [B][Hkv] arrivals per (sequence, KV head), 0 on entry
    int num_kv_heads;
    // FP8 (E4M3) cache only: per-tensor scales (k_scale is also folded into scale_log2)
    float k_scale;
    float v_scale;
#ifdef PA_TEST_HOOKS
    // Test builds only (libpa_test.so): the producer of CTA test_cta (linear
    // index, -1: none) issues no tile from test_tile on, and every pipeline
    // wait gives up after test_wait_limit_ns, so a test can make the
    // consumers' bounded waits run out without a copy in flight.
    int test_cta;
    int test_tile;
    unsigned long long test_wait_limit_ns;
#endif
};

// Work-balanced fused step (balanced.cu): one wave of the fused step's CTAs,
// every consumer warp streaming an equal contiguous range of the (sequence,
// KV head, tile) order.
struct BalancedParams {
    const void* q;
    const int32_t* block_tables;
    const int32_t* context_lens;
    void* out;
    int* err;
    float scale_log2;
    int num_q_heads;
    int group;
    int max_blocks_per_seq;
    int block_size;
    int64_t num_blocks;
    const void* k_new;
    const void* v_new;
    const int64_t* slot_mapping;
    void* k_cache;
    void* v_cache;
    int* counters;                 // [B][Hkv] pieces finished, 0 on entry and on exit
    int num_kv_heads;
    float k_scale;
    float v_scale;
    int num_seqs;
    int num_warps;                 // consumer warps of the grid
    float* rec_o;                  // [R][G][D] partial outputs, R = num_warps + B * Hkv
    float* rec_m;                  // [R][G]
    float* rec_l;                  // [R][G]
};

cudaError_t launch_balanced(int dtype, int head_dim, bool fp8, const CUtensorMap& tmk,
                            const CUtensorMap& tmv, const BalancedParams& p, int num_ctas,
                            cudaStream_t stream);

// Byte copies by SMs (stage_copy.cu): n16 16-byte vectors.
cudaError_t launch_copy16(void* dst, const void* src, size_t n16, cudaStream_t stream);

// Decode kernel modes.
constexpr int kModeSingle = 0;   // one CTA per (sequence, KV head), final output
constexpr int kModeSplit = 1;    // one CTA per partition, partial outputs
constexpr int kModeStep = 2;     // split + cache write of the new token + in-kernel merge

struct ReduceParams {
    const float* tmp_out;
    const float* max_logits;
    const float* exp_sums;
    const int32_t* context_lens;
    void* out;
    int* err;
    int num_q_heads;
    int partition_tokens;
    int max_parts;
    int max_context;               // max_blocks_per_seq * block_size (clamp bound)
};

// Kernel launchers (kernels live in their own translation units).
cudaError_t launch_decode(int dtype, int head_dim, int mode, const CUtensorMap& tmk,
                          const CUtensorMap& tmv, const DecodeParams& p, dim3 grid,
                          cudaStream_t stream);
// Same over an FP8 (E4M3) cache; head_dim 128 only.
cudaError_t launch_decode_fp8(int dtype, int mode, const CUtensorMap& tmk,
                              const CUtensorMap& tmv, const DecodeParams& p, dim3 grid,
                              cudaStream_t stream);
cudaError_t launch_reshape_and_cache_fp8(int dtype, const void* k, const void* v,
                                         const int64_t* slots, void* kc, void* vc,
                                         int64_t num_tokens, int64_t num_slots, int row_elems,
                                         float k_scale, float v_scale, int* err,
                                         cudaStream_t stream);
cudaError_t launch_reduce(int dtype, int head_dim, const ReduceParams& p, int num_seqs,
                          cudaStream_t stream);
cudaError_t launch_reshape_and_cache(const void* k, const void* v, const int64_t* slots,
                                     void* kc, void* vc, int64_t num_tokens,
                                     int64_t num_slots, int row_bytes, int* err,
                                     cudaStream_t stream);

cudaError_t launch_copy_blocks(const void* k_src, const void* v_src, int64_t src_blocks,
                               void* k_dst, void* v_dst, int64_t dst_blocks,
                               const int64_t* mapping, int64_t num_pairs, int64_t block_bytes,
                               int* err, cudaStream_t stream);

// Sets the value pa_last_cuda_error() reports on this host thread.
void record_cuda_error(int cuda_error);

// The calling thread's current CUDA context (cuCtxGetCurrent; null if none).
cudaError_t current_context(void** ctx);

// Argument checks of pa_decode_split + pa_reduce on a 16-bit cache, apart
// from the workspace pointers: PA_OK or the status those entry points return.
int check_split_request(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, const int32_t* context_lens,
                        int32_t partition_size, int32_t max_num_partitions, const void* out,
                        const pa_shape* shp);

}  // namespace pa
