/*
 * pkd.h -- C ABI of the GB300 (sm_103a) paged-KV decode attention library.
 *
 * Operations (all from the vLLM pull-request pages the library is built on):
 *
 *  - pkd_paged_decode_attention: decode-phase attention over a paged KV
 *    cache, the operation vLLM calls single_query_cached_kv_attention
 *    ("Optimizes the single_query_cached_kv_attention kernel", pull request
 *    420).  For every sequence s and query head h,
 *        out[s,h,:] = softmax_t(scale * q[s,h,:] . K_s[t,:]) @ V_s[t,:]
 *    over t < context_lens[s], where
 *        K_s[t] = key_cache[block_tables[s, t / block_size], t % block_size, kv(h), :]
 *    and kv(h) = h / (num_heads / num_kv_heads): contiguous groups of query
 *    heads share one KV head, as in the head mapping of "Optimize MQA
 *    Kernel" (pull request 452), so MHA, GQA and MQA are one call.  Long
 *    contexts at small batch are cut into partitions whose partial results
 *    are merged by a log-sum-exp reduction (the split-context form behind
 *    the "Paged attention V2" column of the kernel-latency tables in
 *    "[Performance] Support MQA/GQA in decode phase by using
 *    FlashAttention", pull request 2744).
 *
 *  - pkd_paged_prefill_attention: several new query tokens per sequence
 *    (a prefill chunk, with or without a cached prefix) attending causally
 *    over the same paged cache; the review comments of pull request 2744
 *    note that the KV-cache attention kernel serves prefill as well.
 *
 *  - pkd_gather_cached_kv: copies the cached K/V rows of the slots listed in
 *    a slot mapping into contiguous [num_tokens, num_heads, head_size]
 *    tensors ("Memcpy kernel for flash attention", pull request 29).
 *
 *  - pkd_reshape_and_cache: the inverse copy, storing new tokens' K/V rows
 *    into their cache slots (the cache_ops.cache step named in the notes of
 *    pull request 2744).
 *
 * Conventions shared by every entry point
 *  - Every tensor argument is a DEVICE pointer owned by the caller, dense
 *    row-major (C order), 16-byte aligned.  16-bit values are IEEE binary16
 *    (PKD_FP16) or bfloat16 (PKD_BF16) bit patterns.
 *  - Cache layout: key_cache and value_cache are
 *    [num_blocks][block_size][num_kv_heads][head_size].  A slot is
 *    block_id * block_size + offset.
 *  - The library allocates no memory and never synchronises the host.  Work
 *    is enqueued on `stream` (a cudaStream_t passed as void*; NULL is the
 *    legacy default stream) in stream order.
 *  - Host-detectable errors return a status before anything is launched.
 *    PKD_ERR_CUDA means a launch failed; pkd_last_error() describes it.
 *  - Data-dependent errors (bad block ids, slots or lengths) cannot be seen
 *    on the host; kernels OR a PKD_DEV_* bit into *device_status (a device
 *    uint32_t, may be NULL) and write the documented fallback output.  The
 *    caller reads the word back whenever it chooses.
 */
#ifndef PKD_H_
#define PKD_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKD_API __attribute__((visibility("default")))
#else
#define PKD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkd_status {
  PKD_OK = 0,
  PKD_ERR_NULL = 1,         /* a required pointer is NULL */
  PKD_ERR_SHAPE = 2,        /* sizes inconsistent or out of range */
  PKD_ERR_UNSUPPORTED = 3,  /* head_size / block_size / dtype not compiled in */
  PKD_ERR_WORKSPACE = 4,    /* workspace missing or smaller than required */
  PKD_ERR_ALIGN = 5,        /* a tensor pointer is not 16-byte aligned */
  PKD_ERR_CUDA = 6,         /* a CUDA runtime call or launch failed */
  PKD_ERR_DEVICE = 7        /* the current device is not an sm_103 GPU */
} pkd_status;

typedef enum pkd_dtype { PKD_FP16 = 0, PKD_BF16 = 1 } pkd_dtype;

/* Bits OR-ed into *device_status by the kernels. */
#define PKD_DEV_BAD_BLOCK 1u /* a referenced block id is outside [0, num_blocks) */
#define PKD_DEV_BAD_SLOT 2u  /* a slot is outside [0, num_blocks * block_size) */
#define PKD_DEV_BAD_LEN 4u   /* context_lens[s] < 0, > max_context_len or > table */
#define PKD_DEV_TIMEOUT 8u   /* a bounded wait inside a kernel gave up */

/* Decode kernel families, as reported by pkd_decode_plan(). */
#define PKD_PATH_SIMT 0   /* CUDA-core path (query-group size below 4) */
#define PKD_PATH_TC 1     /* tcgen05 tensor-core path with TMA staging */
#define PKD_PATH_TC_CLUSTER 2 /* the same, its context partitions merged inside
                                 thread-block clusters: no workspace, one launch */
#define PKD_PATH_TC_STREAM 3  /* the tensor-core kernel in stream form: one CTA per
                                 SM, each taking an equal contiguous share of all
                                 128-token tiles; the (sequence, KV head) runs cut
                                 at a share's edges are merged by a second launch */

/* partition_size value that asks for the stream form (tensor-core path,
 * num_seqs <= 1024); the call returns PKD_ERR_UNSUPPORTED where it cannot
 * be used. */
#define PKD_PARTITION_STREAM (-1)

/*
 * Launch plan of pkd_paged_decode_attention for the given sizes on the
 * CURRENT device (same size rules as that call).  partition_size = 0 lets
 * the library choose; a positive value (a multiple of 64 tokens) forces
 * that partition length; PKD_PARTITION_STREAM forces the stream form, which
 * reports a partition length of 128 and one partition.  Outputs
 * (any may be NULL): the partition length in tokens, the number of
 * partitions (1 = no split, no reduction launch), the kernel family, and the
 * workspace bytes the call needs (0 when unsplit, and for
 * PKD_PATH_TC_CLUSTER, whose split is merged inside the one launch).  The
 * tensor-core path merges a split inside thread-block clusters when it has
 * at most 16 partitions and the clusters of all (sequence, KV head) pairs fit
 * on the device at once.  It takes the stream form (workspace: 2 partial
 * rows per SM and query head of a group, plus the tile prefix) when that
 * form's estimated time, which assumes every sequence at max_context_len,
 * is lower.  Pure host arithmetic plus cached device-attribute
 * and occupancy queries; allocates nothing.
 */
PKD_API pkd_status pkd_decode_plan(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                           int block_size, int max_context_len, int partition_size,
                           int* out_partition_size, int* out_num_partitions, int* out_path,
                           size_t* out_workspace_bytes);

/*
 * Workspace bytes that pkd_paged_decode_attention needs with partition_size
 * 0 (the library's own plan) on the CURRENT device, for any num_kv_heads
 * dividing num_heads and any supported block_size: the largest over those
 * plans, so a buffer of this size serves every such call with these four
 * sizes.  0 when no plan needs a workspace, and also when the sizes are
 * invalid or the current device is not an sm_103 GPU (pkd_decode_plan
 * reports those as errors, and gives the exact size for one configuration).
 * Allocates nothing.
 */
PKD_API size_t pkd_decode_workspace_bytes(int num_seqs, int num_heads, int head_size,
                                          int max_context_len);

/*
 * Decode attention over a paged KV cache.
 *   out           [num_seqs][num_heads][head_size]            16-bit, written
 *   q             [num_seqs][num_heads][head_size]            16-bit
 *   key_cache,
 *   value_cache   [num_blocks][block_size][num_kv_heads][head_size] 16-bit
 *   block_tables  [num_seqs][max_blocks_per_seq] int32; entries past
 *                 ceil(context_lens[s] / block_size) are ignored (their
 *                 values do not matter; max_blocks_per_seq * block_size
 *                 must stay below 2^31 - 2^16)
 *   context_lens  [num_seqs] int32, each in [0, max_context_len]
 *   max_context_len  host-side upper bound of context_lens (sizes the grid)
 *   num_heads % num_kv_heads == 0;  head_size in {64, 128};
 *   block_size a power of two in [8, 256];  1 <= num_seqs <= 65535
 *   scale         logit multiplier (1/sqrt(head_size) for standard attention)
 *   partition_size  0 = library choice, PKD_PARTITION_STREAM = stream form,
 *                 else a multiple of 64 tokens
 *   workspace     device scratch of >= the plan's workspace bytes (may be
 *                 NULL when that is 0); its contents on entry do not matter
 *                 and are clobbered
 *   device_status optional device uint32_t for PKD_DEV_* bits
 * Results are rounded to nearest-even from fp32 accumulation.  A sequence
 * with context_lens[s] == 0 yields zeros.  A sequence with an invalid length
 * or a referenced block id outside [0, num_blocks) yields zeros and sets the
 * matching PKD_DEV_* bit.
 */
PKD_API pkd_status pkd_paged_decode_attention(void* out, const void* q, const void* key_cache,
                                      const void* value_cache, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* context_lens,
                                      int max_context_len, int num_seqs, int num_heads,
                                      int num_kv_heads, int head_size, int block_size,
                                      int num_blocks, float scale, pkd_dtype dtype,
                                      int partition_size, void* workspace,
                                      size_t workspace_bytes, uint32_t* device_status,
                                      void* stream);

/*
 * pkd_paged_decode_attention with an optional ALiBi bias.  Same arguments,
 * plus alibi_slopes: NULL, or a device array [num_heads] of float slopes
 * (4-byte aligned).  With slopes, the logit of token t of sequence s for
 * query head h becomes
 *     scale * q[s,h,:] . K_s[t,:] + alibi_slopes[h] * (t - context_lens[s] + 1),
 * the linear position bias that "Optimize MQA Kernel" (vLLM pull request
 * 452) names as combining with MQA; the FlashAttention pull request's
 * kernel-latency runs use it switched off.  NULL gives exactly
 * pkd_paged_decode_attention.
 */
PKD_API pkd_status pkd_paged_decode_attention_ex(
    void* out, const void* q, const void* key_cache, const void* value_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int num_seqs, int num_heads, int num_kv_heads, int head_size,
    int block_size, int num_blocks, float scale, const float* alibi_slopes, pkd_dtype dtype,
    int partition_size, void* workspace, size_t workspace_bytes, uint32_t* device_status,
    void* stream);

/* Size of the scratch array built into the library for
 * pkd_paged_decode_attention_static_ws (16 MiB per GPU that loads it). */
#define PKD_STATIC_WORKSPACE_BYTES (16u * 1024u * 1024u)

/*
 * Decode attention for callers that cannot allocate device memory.  (The
 * vLLM pages have no counterpart: this is an interface addition.)
 *
 * Same arguments, results and errors as pkd_paged_decode_attention, minus
 * the workspace: the split-context scratch comes from an array of
 * PKD_STATIC_WORKSPACE_BYTES bytes compiled into the library, so the call
 * allocates nothing and needs nothing from the caller beyond inputs and
 * outputs.  It serves code that must not call cudaMalloc while it runs -- a
 * serving loop that may never touch the allocator, a runtime whose device
 * memory is pre-carved by another owner, an operator plugin handed only its
 * input and output pointers.
 *   - Returns PKD_ERR_WORKSPACE, launching nothing, when the launch plan
 *     (pkd_decode_plan with the same sizes) needs more scratch than
 *     PKD_STATIC_WORKSPACE_BYTES; pass a larger partition_size, or use
 *     pkd_paged_decode_attention with a caller-provided workspace.
 *   - The first call on each device, with that device current, looks up the
 *     array's device address once (cudaGetSymbolAddress); make that first
 *     call before any stream capture.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents; nothing in it needs to start at zero.  Calls that
 *     overlap on the GPU (e.g. on two streams at once) race on it: order them.
 *   - Every GPU that loads the library holds the array until process exit.
 */
PKD_API pkd_status pkd_paged_decode_attention_static_ws(
    void* out, const void* q, const void* key_cache, const void* value_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int num_seqs, int num_heads, int num_kv_heads, int head_size,
    int block_size, int num_blocks, float scale, pkd_dtype dtype, int partition_size,
    uint32_t* device_status, void* stream);

/*
 * Prefill over a paged KV cache: each sequence brings a chunk of new query
 * tokens whose K/V rows are already in its cache as its LAST tokens (store
 * them first with pkd_reshape_and_cache), and each query attends causally
 * to the cache up to its own position.  With n_s = query_start[s+1] -
 * query_start[s] and L_s = context_lens[s] (which counts the chunk), query
 * i of sequence s (packed row r = query_start[s] + i) sits at position
 * p = L_s - n_s + i and
 *     out[r,h,:] = softmax_{t <= p}(scale * q[r,h,:] . K_s[t,:] + bias) @ V_s[t,:]
 * with K_s, V_s and the query-head -> KV-head groups exactly as in
 * pkd_paged_decode_attention; bias = alibi_slopes[h] * (t - p) when
 * alibi_slopes is not NULL.  n_s = 1 is decode; n_s = L_s is a prompt
 * without prefix.
 *   out, q          [num_query_tokens][num_heads][head_size] 16-bit
 *   query_start     [num_seqs + 1] int32, non-decreasing from 0, with
 *                   query_start[num_seqs] == num_query_tokens (rows past
 *                   query_start[num_seqs] are not written; a sequence whose
 *                   rows fall outside [0, num_query_tokens) is skipped and
 *                   sets PKD_DEV_BAD_LEN)
 *   max_query_len   host-side upper bound of n_s (sizes the grid)
 *   other arguments as for pkd_paged_decode_attention_ex; head_size must be
 *   128 and num_heads / num_kv_heads at most 64 (else PKD_ERR_UNSUPPORTED).
 * One launch of the tensor-core kernel (tcgen05 MMAs over (query, head)
 * columns, up to 64 per work unit); no workspace.  A chunk with
 * n_s > L_s or n_s > max_query_len, or an invalid L_s (as for decode),
 * gives zero rows and sets PKD_DEV_BAD_LEN.  A query whose window t <= p
 * references a block id outside [0, num_blocks) gives a zero row and sets
 * PKD_DEV_BAD_BLOCK; the queries before that block are unaffected.
 */
PKD_API pkd_status pkd_paged_prefill_attention(
    void* out, const void* q, const void* key_cache, const void* value_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    const int32_t* query_start, int num_query_tokens, int max_query_len, int max_context_len,
    int num_seqs, int num_heads, int num_kv_heads, int head_size, int block_size, int num_blocks,
    float scale, const float* alibi_slopes, pkd_dtype dtype, uint32_t* device_status,
    void* stream);

/*
 * gather_cached_kv: key_out[t] = key_cache[slot / block_size][slot % block_size]
 * and value_out[t] likewise, slot = slot_mapping[t], bit for bit.
 *   key_out, value_out        [num_tokens][num_heads][head_size] 16-bit, written
 *   key_cache, value_cache    [num_blocks][block_size][num_heads][head_size]
 *   slot_mapping              [num_tokens] int64
 * num_tokens may be 0 (nothing is launched).  A slot outside
 * [0, num_blocks * block_size) gives zero rows and sets PKD_DEV_BAD_SLOT.
 * head_size must be a multiple of 8; any block_size >= 1.
 */
PKD_API pkd_status pkd_gather_cached_kv(void* key_out, void* value_out, const void* key_cache,
                                const void* value_cache, const int64_t* slot_mapping,
                                int num_tokens, int num_heads, int head_size, int block_size,
                                int num_blocks, pkd_dtype dtype, uint32_t* device_status,
                                void* stream);

/*
 * reshape_and_cache: key_cache[slot / block_size][slot % block_size] = key[t]
 * and the same for value, slot = slot_mapping[t], bit for bit.
 *   key, value                [num_tokens][num_heads][head_size] 16-bit
 *   key_cache, value_cache    [num_blocks][block_size][num_heads][head_size], updated
 *   slot_mapping              [num_tokens] int64
 * A negative slot marks a token that is not stored (no status bit).  A slot
 * at or past num_blocks * block_size is not stored and sets PKD_DEV_BAD_SLOT.
 * Two tokens with the same slot race; the caller must not do that.
 */
PKD_API pkd_status pkd_reshape_and_cache(const void* key, const void* value, void* key_cache,
                                 void* value_cache, const int64_t* slot_mapping, int num_tokens,
                                 int num_heads, int head_size, int block_size, int num_blocks,
                                 pkd_dtype dtype, uint32_t* device_status, void* stream);

/*
 * Self-test of failure detection without a GPU fault.  Every kernel's waits
 * are bounded: a wait that gives up ORs PKD_DEV_TIMEOUT into device_status
 * and the kernel returns.  This launches one thread that waits, through that
 * same routine, on a shared-memory barrier nothing arrives on, for limit_ns
 * nanoseconds (1e3 .. 1e9); it then sets PKD_DEV_TIMEOUT in *device_status
 * (a device uint32_t) and returns, leaving the context usable.  Host
 * errors: PKD_ERR_NULL without device_status, PKD_ERR_SHAPE for a limit out
 * of range, both before any launch.
 */
PKD_API pkd_status pkd_selftest_bounded_wait(uint32_t* device_status, long long limit_ns,
                                             void* stream);

/* Static text for a status code. */
PKD_API const char* pkd_status_string(pkd_status status);

/* Text of the last PKD_ERR_CUDA raised on this host thread ("" if none). */
PKD_API const char* pkd_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
PKD_API int pkd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKD_H_ */
