// Chunked-prefill kernels' parameters and launchers (prefill.cu: mma.sync;
// prefill_tc.cu: tcgen05), apart from the decode declarations so that the
// two families' sources change independently.
#pragma once

#include "pa_internal.h"

namespace pa {

// Paged prefill (prefill.cu).
struct PrefillParams {
    const void* q;                 // [T][Hq][D]
    void* out;                     // [T][Hq][D]
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* query_start;    // [B + 1]
    int* err;
    float scale_log2;
    int num_q_heads;
    int group;
    int max_blocks_per_seq;
    int block_size;
    int64_t num_blocks;
    // tcgen05 kernel only: the order in which its persistent CTAs deal out
    // the (sequence, chunk) items, num_seqs * max_chunks entries of b *
    // max_chunks + chunk (-1: none), longest first; null: later chunks (more
    // keys) first
    const int32_t* sched;
    int max_chunks;                // chunk slots per sequence
    int num_seqs;
};

cudaError_t launch_prefill(int dtype, int head_dim, const CUtensorMap& tmk,
                           const CUtensorMap& tmv, const PrefillParams& p, dim3 grid,
                           cudaStream_t stream);

// tcgen05 chunked prefill (prefill_tc.cu): head_dim 128, groups of 1, 2, 4, 8,
// a positive softmax scale.
bool prefill_tc_supported(int head_dim, int group, float scale);
// Chunk slots per sequence: query tokens per work unit are 128 / group.
int prefill_tc_chunks(int group, int max_query_len);
// One CTA: writes the order of the num_seqs * max_chunks items, longest
// (most key tiles) first, to sched (p.sched is ignored).
cudaError_t launch_prefill_tc_plan(const PrefillParams& p, int32_t* sched, cudaStream_t stream);
cudaError_t launch_prefill_tc(int dtype, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              const PrefillParams& p, int num_kv_heads, cudaStream_t stream);

}  // namespace pa
