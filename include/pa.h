/*
 * pa.h -- C ABI of the paged decode attention library (libpa.so).
 *
 * The operation (from the pages on vLLM / PagedAttention):
 *   - The KV cache is split into fixed-size blocks (16 tokens by default) that
 *     may sit anywhere in a preallocated physical pool; a per-request block
 *     table maps logical block j to its physical block (techfeed summary of
 *     ngrok's "Serving models at scale with vLLM", section on PagedAttention;
 *     youngju.dev "vLLM inference optimization", section "PagedAttention").
 *   - A new token's K and V go to slot (last block, count % block_size)
 *     (youngju.dev post, PagedAttentionManager.append_token).
 *   - Decode attention follows the table, gathering K and V while it computes
 *     (ta-paperlens "LLM serving from scratch", section on fragmentation and
 *     PagedAttention).
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 * Layouts are row-major and contiguous; every pointer marked (device) is
 * CUDA device memory (or managed memory) of the current device:
 *   q, out          [num_seqs][num_q_heads][head_dim]                 T
 *   k, v (new)      [num_tokens][num_kv_heads][head_dim]              T
 *   k_cache,v_cache [num_blocks][block_size][num_kv_heads][head_dim]  T
 *   block_tables    [num_seqs][max_blocks_per_seq]                    int32
 *   context_lens    [num_seqs]                                        int32
 *   slot_mapping    [num_tokens]                                      int64
 * where T is fp16 or bf16 (pa_shape.dtype).  Query head h reads KV head
 * h / (num_q_heads / num_kv_heads).  context_lens[b] counts every token of
 * sequence b including the one just written; token i lives at offset
 * i % block_size of physical block block_tables[b][i / block_size].
 * Attention is softmax(scale * q . K^T) . V with fp32 accumulation; outputs
 * are rounded to nearest-even into T.  An empty context gives zeros.
 *
 * Ownership: the caller owns every buffer, including split workspaces.  The
 * library allocates nothing, frees nothing and never synchronises: work is
 * enqueued on `stream` (a cudaStream_t passed as void*; NULL = the legacy
 * default stream) and the call returns once it is enqueued.
 *
 * Errors: arguments are validated on the host before anything is enqueued;
 * a failed check returns a non-zero pa_status and launches nothing.  A
 * failed launch returns PA_ERR_CUDA (pa_last_cuda_error gives the code).
 * Device-side values are bounded rather than trusted: a context length is
 * clamped to [0, max_blocks_per_seq * block_size]; a physical block id
 * outside [0, num_blocks) reads as zeros (never out of the pool); a slot
 * outside the pool is skipped.  Those events, and any wait in a kernel that
 * ran past its time limit, set bits of a device error word read with
 * pa_read_device_errors.
 *
 * Supported shapes: head_dim 64 or 128; block_size 16 or 32; 1 <= num_q_heads /
 * num_kv_heads <= 8; every device pointer 16-byte aligned.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, inconsistent shape */
    PA_ERR_UNSUPPORTED = 2,   /* valid but not built: head_dim, block_size, group */
    PA_ERR_WORKSPACE = 3,     /* split workspace too small for the request */
    PA_ERR_CUDA = 4           /* a CUDA call failed; see pa_last_cuda_error */
} pa_status;

typedef enum { PA_FP16 = 0, PA_BF16 = 1 } pa_dtype;

/* Device error word bits (pa_read_device_errors). */
#define PA_DEVERR_WAIT_TIMEOUT   0x1  /* a pipeline wait gave up after ~1 s */
#define PA_DEVERR_BAD_CONTEXT    0x2  /* a context length was clamped */
#define PA_DEVERR_BAD_SLOT       0x4  /* a slot past the pool was skipped */

typedef struct {
    int32_t num_seqs;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t block_size;
    int32_t max_blocks_per_seq;
    int64_t num_blocks;
    int32_t dtype;            /* pa_dtype */
    int32_t reserved;         /* must be 0 */
} pa_shape;

/*
 * reshape_and_cache: write each new token's K and V into its cache slot.
 * For t < num_tokens with s = slot_mapping[t] (device):
 *   s < 0                       -> padding, nothing written;
 *   0 <= s < num_blocks*block_size
 *       -> k_cache[s / block_size][s % block_size][:][:] = k[t][:][:],
 *          v_cache likewise (bit copy);
 *   otherwise                   -> skipped, PA_DEVERR_BAD_SLOT set.
 * (youngju.dev post, PagedAttentionManager.append_token.)
 * k, v, slot_mapping, k_cache, v_cache: device.  Uses shp->num_kv_heads,
 * head_dim, block_size, num_blocks and dtype; num_seqs may differ from
 * num_tokens and is ignored.  num_tokens == 0 enqueues nothing.
 */
int pa_reshape_and_cache(const void* k, const void* v, const int64_t* slot_mapping,
                         void* k_cache, void* v_cache, int64_t num_tokens,
                         const pa_shape* shp, void* stream);

/*
 * pa_decode: single-pass paged decode attention, one query token per sequence
 * (ta-paperlens page, PagedAttention paragraph): for every b, h
 *   out[b][h][:] = sum_i softmax_i(scale * q[b][h] . K_i) V_i,  i < context_lens[b].
 * One CTA walks the whole context of a (sequence, KV head) and serves the
 * group of query heads that share the KV head.
 * q, k_cache, v_cache, block_tables, context_lens, out: device.
 */
int pa_decode(const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, const int32_t* context_lens, float scale,
              void* out, const pa_shape* shp, void* stream);

/*
 * Bytes of one contiguous split workspace for pa_decode_split / pa_reduce:
 * [tmp_out][max_logits][exp_sums], each part rounded up to 256 bytes, with
 * max_num_partitions = ceil(max_context_len / partition_size).
 * Returns 0 for invalid arguments.
 */
size_t pa_split_workspace_size(const pa_shape* shp, int32_t max_context_len,
                               int32_t partition_size);

/*
 * pa_decode_split: the context of each sequence is cut into partitions of
 * partition_size tokens (a multiple of block_size); partition s covers
 * tokens [s*P, min((s+1)*P, L_b)).  For each (b, h, s) with s*P < L_b and
 * s < max_num_partitions it writes, in fp32:
 *   max_logits[b][h][s]   = m_s = max_i scale * q . K_i
 *   exp_sums[b][h][s]     = l_s = sum_i exp(scale * q . K_i - m_s)
 *   tmp_out[b][h][s][:]   = sum_i exp(scale * q . K_i - m_s) V_i / l_s
 * Partitions at or past the context end are not written.  Tokens at or past
 * max_num_partitions * partition_size are not attended: the caller sizes
 * max_num_partitions >= ceil(max_b L_b / partition_size).
 * tmp_out [B][Hq][max_num_partitions][D], max_logits and exp_sums
 * [B][Hq][max_num_partitions]: device, fp32, 16-byte aligned.
 * (Context split and log-sum-exp merge are not in the pages; they follow
 * the split-context decoding used for long contexts.)
 */
int pa_decode_split(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, const int32_t* context_lens, float scale,
                    int32_t partition_size, int32_t max_num_partitions,
                    float* tmp_out, float* max_logits, float* exp_sums,
                    const pa_shape* shp, void* stream);

/*
 * pa_reduce: log-sum-exp merge of pa_decode_split's partitions.  For each
 * (b, h) with S_b = min(ceil(L_b / P), max_num_partitions):
 *   M = max_s m_s,  w_s = l_s * exp(m_s - M),
 *   out[b][h][:] = sum_s w_s tmp_out[b][h][s][:] / sum_s w_s   (zeros if S_b = 0).
 * tmp_out, max_logits, exp_sums, context_lens, out: device.
 */
int pa_reduce(const float* tmp_out, const float* max_logits, const float* exp_sums,
              const int32_t* context_lens, int32_t partition_size,
              int32_t max_num_partitions, void* out, const pa_shape* shp, void* stream);

/*
 * pa_decode_step_balanced: the fused layer-step of pa_decode_step (same
 * inputs, same results) with the work balanced over one wave of CTAs instead
 * of one CTA per context partition: the 16-token tiles of all (sequence,
 * KV head) pairs, in order, are dealt out in equal contiguous ranges to the
 * consumer warps of the grid, each CTA's TMA producer warp serving its two
 * consumers; a warp's range may cover the end of one sequence and the start
 * of the next, and pieces of one (sequence, KV head) are merged
 * (log-sum-exp) by the warp that finishes last.  Suited to batches of many
 * short or ragged contexts.
 * workspace: device memory of at least pa_balanced_workspace_size(shp)
 * bytes, 16-byte aligned, all zero before the first call (it holds
 * per-(sequence, KV head) counters that every call leaves at zero; zero it
 * again after a PA_DEVERR_WAIT_TIMEOUT).  Calls that overlap on the GPU must
 * not share a workspace.  Other arguments and errors as pa_decode_step.
 * One launch.
 */
size_t pa_balanced_workspace_size(const pa_shape* shp);
int pa_decode_step_balanced(const void* q, const void* k, const void* v,
                            const int64_t* slot_mapping, void* k_cache, void* v_cache,
                            const int32_t* block_tables, const int32_t* context_lens, float scale,
                            void* workspace, size_t workspace_bytes, void* out,
                            const pa_shape* shp, void* stream);

/*
 * FP8 KV cache.  The pages name the KV-cache data type as a knob that, like
 * weight quantisation, shrinks the KV pool so that more requests fit
 * (ta-paperlens page, --quantization / --kv-cache-dtype; youngju.dev post,
 * quantisation section).  Here the cache holds OCP E4M3 codes (1 byte per
 * element, [num_blocks][block_size][num_kv_heads][head_dim] bytes) with one
 * scale per tensor: element = e4m3(code) * k_scale (K) or * v_scale (V).
 * q, k, v (new tokens) and out keep the 16-bit type of shp->dtype.
 * head_dim must be 128 (else PA_ERR_UNSUPPORTED); scales must be finite and
 * > 0 (else PA_ERR_INVALID_ARG).  Otherwise these mirror the 16-bit entry
 * points, argument for argument, with the scales added.
 *
 * pa_reshape_and_cache_fp8: code = E4M3 of x / k_scale (x / v_scale), the
 * quotient in fp32, rounded to nearest even, saturating at +-448.
 */
int pa_reshape_and_cache_fp8(const void* k, const void* v, const int64_t* slot_mapping,
                             void* k_cache, void* v_cache, int64_t num_tokens, float k_scale,
                             float v_scale, const pa_shape* shp, void* stream);

/* pa_decode over an E4M3 cache. */
int pa_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens, float scale,
                  float k_scale, float v_scale, void* out, const pa_shape* shp, void* stream);

/* pa_decode_split over an E4M3 cache (merge the partitions with pa_reduce). */
int pa_decode_split_fp8(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, const int32_t* context_lens, float scale,
                        float k_scale, float v_scale, int32_t partition_size,
                        int32_t max_num_partitions, float* tmp_out, float* max_logits,
                        float* exp_sums, const pa_shape* shp, void* stream);

/* pa_decode_step over an E4M3 cache (the same memory rules, pinned host
 * inputs and output included): the new token is quantised as in
 * pa_reshape_and_cache_fp8 and attention reads the quantised values. */
int pa_decode_step_fp8(const void* q, const void* k, const void* v, const int64_t* slot_mapping,
                       void* k_cache, void* v_cache, const int32_t* block_tables,
                       const int32_t* context_lens, float scale, float k_scale, float v_scale,
                       int32_t partition_size, int32_t max_num_partitions, float* tmp_out,
                       float* max_logits, float* exp_sums, int32_t* counters, void* out,
                       const pa_shape* shp, void* stream);

/* pa_decode_step_balanced over an E4M3 cache. */
int pa_decode_step_balanced_fp8(const void* q, const void* k, const void* v,
                                const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                const int32_t* block_tables, const int32_t* context_lens,
                                float scale, float k_scale, float v_scale, void* workspace,
                                size_t workspace_bytes, void* out, const pa_shape* shp,
                                void* stream);

/*
 * pa_prefill: paged prefill / chunked-prefill attention.  Sequence b holds
 * L_b = context_lens[b] tokens in the cache, the last C_b = query_start[b+1]
 * - query_start[b] of which are new in this step (written beforehand with
 * pa_reshape_and_cache).  New token i of b sits at position p = L_b - C_b + i
 * and attends causally:
 *   out[query_start[b] + i][h][:] = sum_{j <= p} softmax_j(scale q.K_j) V_j
 * (ta-paperlens page, prefill vs decode and chunked prefill; techfeed
 * summary, chunked prefill of long prompts).  A one-token chunk is a decode.
 * q, out: [total_tokens][num_q_heads][head_dim] with total_tokens =
 * query_start[num_seqs]; query_start int32 [num_seqs + 1], non-decreasing,
 * from 0; max_query_len >= every C_b (it sizes the grid: query tokens past
 * 16 * ceil(max_query_len / 16) are not computed).  C_b > L_b is clamped to
 * L_b and flagged (PA_DEVERR_BAD_CONTEXT).  All pointers device.
 */
int pa_prefill(const void* q, const void* k_cache, const void* v_cache,
               const int32_t* block_tables, const int32_t* context_lens,
               const int32_t* query_start, float scale, int32_t max_query_len, void* out,
               const pa_shape* shp, void* stream);

/*
 * pa_prefill_ws: pa_prefill with a workspace in which a one-CTA plan kernel
 * orders the tcgen05 kernel's (sequence, chunk) work items by the number of
 * key tiles they read, longest first, so that the longest start first and
 * the SMs finish together (the kernel's persistent CTAs, one per SM, deal
 * that order out in a snake; pa_prefill, without one, takes each sequence's
 * chunks last-first: later chunks read more keys).  The pages describe
 * prefill cost growing with the square of the prompt length (ta-paperlens
 * page, the quadratic cost of prefill); the ordering itself is this
 * library's.  workspace: device memory of at least
 * pa_prefill_workspace_size(shp, max_query_len) bytes, 16-byte aligned, no
 * initial contents, owned by the caller; calls that overlap on the GPU must
 * not share it.  A size of 0 (the mma.sync kernel is taken) accepts a null
 * workspace, which otherwise also falls back to pa_prefill's order.  Too
 * small or misaligned: PA_ERR_INVALID_ARG.  Two launches when the tcgen05
 * kernel is taken with a workspace, else one.  Results are bitwise the same
 * as pa_prefill's.
 */
size_t pa_prefill_workspace_size(const pa_shape* shp, int32_t max_query_len);
int pa_prefill_ws(const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* block_tables, const int32_t* context_lens,
                  const int32_t* query_start, float scale, int32_t max_query_len,
                  void* workspace, size_t workspace_bytes, void* out, const pa_shape* shp,
                  void* stream);

/*
 * pa_prefill_mma: the same operation, arguments and errors as pa_prefill,
 * always on the mma.sync kernel (16 query tokens per CTA, any group size and
 * head_dim 64 or 128).  pa_prefill takes the tcgen05 kernel (128 query rows
 * per CTA, accumulators in tensor memory) when head_dim is 128, the group
 * size G = Hq / Hkv is 1, 2, 4 or 8, scale > 0 and max_query_len >= 128 / G
 * (a chunk can fill its 128 rows), and this one otherwise.
 */
int pa_prefill_mma(const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* block_tables, const int32_t* context_lens,
                   const int32_t* query_start, float scale, int32_t max_query_len, void* out,
                   const pa_shape* shp, void* stream);

/*
 * pa_copy_async: copy nbytes from src to dst with a short kernel on the
 * stream (SM loads and stores, not a copy-engine transfer).  For a
 * layer-step's small transfers: dst and src may each be device memory or
 * pinned host memory (reached through unified addressing), both 16-byte
 * aligned, nbytes a multiple of 16; the buffers must not overlap.  The launch
 * takes part in programmatic dependent launch like the step kernels, so an
 * upload, a step and a read-back chain without gaps.  No counterpart in the
 * pages: it is the transport of the step's inputs and output.
 */
int pa_copy_async(void* dst, const void* src, size_t nbytes, void* stream);

/*
 * pa_copy_blocks: copy whole physical blocks between two block pools.  For
 * each pair p < num_pairs of block_mapping (int64 [num_pairs][2], device):
 *   src = block_mapping[2p], dst = block_mapping[2p+1],
 *   k_dst[dst][:][:][:] = k_src[src][:][:][:], v_dst likewise (bit copy).
 * Copy-on-write: before a request writes into a block it shares with others
 * (parallel sampling, beam search, a shared prompt), it gets a private copy
 * (tcdigital article, memory sharing for parallel sampling; youngju.dev post,
 * Copy-on-Write prefix sharing) -- src and dst pools are the same pool.
 * Swap: a preempted request's blocks move to CPU memory and back (tcdigital
 * article, --swap-space; ta-paperlens scheduler, preemption) -- one pool is
 * pinned host memory reachable from the device (cudaHostAlloc / registered
 * memory under unified addressing), passed by its device-visible address.
 * Both pools are laid out [num_blocks][block_size][num_kv_heads][head_dim]
 * with shp's block_size, num_kv_heads, head_dim and dtype (shp->num_blocks is
 * not used); src_num_blocks / dst_num_blocks bound the ids.  A pair with an
 * id out of range is skipped and sets PA_DEVERR_BAD_SLOT.  Pairs must not
 * write the same destination block twice, nor read a block another pair
 * writes.  num_pairs <= 65535; num_pairs == 0 enqueues nothing.
 */
int pa_copy_blocks(const void* k_src, const void* v_src, int64_t src_num_blocks, void* k_dst,
                   void* v_dst, int64_t dst_num_blocks, const int64_t* block_mapping,
                   int64_t num_pairs, const pa_shape* shp, void* stream);

/*
 * Size of the device buffer behind pa_decode_static_workspace: 32 MiB,
 * held on every GPU that loads the library until the process exits.
 */
#define PA_STATIC_WORKSPACE_BYTES (32u << 20)

/*
 * pa_decode_static_workspace: pa_decode_split followed by pa_reduce, with the
 * partition workspace (tmp_out, max_logits, exp_sums) taken from a fixed
 * device buffer inside the library instead of from the caller.  It allocates
 * nothing.  The pages have no counterpart: this entry point exists for
 * callers that cannot allocate device memory -- code running inside a host
 * framework that owns the device memory pool (a private cudaMalloc would
 * bypass the pool and may fail once the pool holds the free memory), or a
 * latency-critical loop that cannot take the device-wide synchronisation of
 * cudaMalloc / cudaFree.  The caller passes its inputs and `out` exactly as
 * for pa_decode_split + pa_reduce (same layouts, same device pointers,
 * partition_size a multiple of block_size, max_num_partitions >=
 * ceil(max_b L_b / partition_size)); out [B][Hq][D] receives the merged
 * attention output.
 *
 * Limit: the workspace, laid out [tmp_out][max_logits][exp_sums] with each
 * part rounded up to 256 bytes (4*B*Hq*S*D, then 4*B*Hq*S twice), must fit in
 * PA_STATIC_WORKSPACE_BYTES; larger requests return PA_ERR_WORKSPACE and
 * enqueue nothing.
 *
 * Set-up: the first call on a device (with that device current) looks up the
 * buffer's device address; make that first call before any stream capture.
 * The address belongs to the CUDA context it was looked up in: a call under
 * another context (a driver-API context made current by the caller, or the
 * primary context created anew after cudaDeviceReset) looks it up again, so
 * the first call under each new context must also come before any capture.
 *
 * Sharing: every call on a device uses the same buffer, which keeps the last
 * call's contents (nothing in it needs to start at zero).  Calls whose work
 * overlaps on the GPU -- e.g. issued on two streams without ordering between
 * them -- race on the buffer and corrupt each other's results; order them.
 * Errors: the argument checks of pa_decode_split and pa_reduce run first and
 * give the same statuses; then PA_ERR_WORKSPACE for the limit above.
 */
int pa_decode_static_workspace(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const int32_t* context_lens,
                               float scale, int32_t partition_size,
                               int32_t max_num_partitions, void* out, const pa_shape* shp,
                               void* stream);

/*
 * pa_decode_step: one decode layer-step in a single launch -- the cache write
 * of each sequence's new token followed by split decode attention and the
 * log-sum-exp merge.  Same results as
 *   pa_reshape_and_cache(k, v, slot_mapping, k_cache, v_cache, num_seqs, ...);
 *   pa_decode_split(...); pa_reduce(...);
 * for the decode step the pages describe (youngju.dev post,
 * PagedAttentionManager.append_token, then the table-walking attention of
 * the ta-paperlens page): token b of k, v ([num_seqs][Hkv][D]) is sequence
 * b's newest token, position L_b - 1, and slot_mapping[b] must be that
 * position's slot, block_tables[b][(L_b-1)/bs]*bs + (L_b-1)%bs, or negative
 * (no new token for b: nothing written).  Any other slot is not written and
 * sets PA_DEVERR_BAD_SLOT.  The CTA of each sequence's last partition writes
 * the new token into the cache and uses it directly; the last CTA of each
 * (sequence, KV head) to finish merges its partitions, so no second launch
 * is needed.
 *
 * Workspace: tmp_out, max_logits, exp_sums as for pa_decode_split, plus
 * counters, int32 [num_seqs][num_kv_heads], which must be zero on entry and
 * are zero again when the step has run (set them to zero once after
 * allocation; after a PA_DEVERR_WAIT_TIMEOUT, zero them again).  The merge
 * reads the partition records four at a time from global memory, so any
 * partition count pa_decode_split accepts works.  out [B][Hq][D] receives
 * the attention output.  k_cache, v_cache and the workspace are device memory;
 * q, k, v, slot_mapping, block_tables, context_lens and out may be device
 * memory or pinned host memory that the device reaches through unified
 * addressing (each CTA reads its inputs and writes its output directly, so
 * a step needs no separate upload or read-back; on a Grace-Blackwell node
 * this moves them over the coherent host link).  k, v, out, tmp_out,
 * max_logits, exp_sums 16-byte aligned; errors as pa_decode_split.
 */
int pa_decode_step(const void* q, const void* k, const void* v, const int64_t* slot_mapping,
                   void* k_cache, void* v_cache, const int32_t* block_tables,
                   const int32_t* context_lens, float scale, int32_t partition_size,
                   int32_t max_num_partitions, float* tmp_out, float* max_logits,
                   float* exp_sums, int32_t* counters, void* out, const pa_shape* shp,
                   void* stream);

/* Static description of a status code. */
const char* pa_status_string(int status);

/* cudaError_t of the most recent PA_ERR_CUDA on this host thread (0 if none). */
int pa_last_cuda_error(void);

/*
 * Copy the device error word (PA_DEVERR_* bits accumulated by kernels of this
 * library on the current device) to *flags, then clear it.  Synchronises
 * `stream`.  Returns PA_OK or PA_ERR_CUDA.
 */
int pa_read_device_errors(int32_t* flags, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
