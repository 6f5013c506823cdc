/*
 * pa.h - C ABI of the GB300 (sm_103a) paged-KV attention library (libpa.so).
 *
 * The KV cache is a pool of fixed-size physical blocks of 16 tokens placed anywhere in
 * device memory; a sequence reaches its blocks through a block table that maps logical
 * block i to a physical block id ("vLLM Internals: From PagedAttention to Removing
 * PagedAttention", section 1.1; "My Understanding of vLLM and PagedAttention", sections
 * "Logical Blocks", "Physical Blocks" and "Block Table"). The table is a dense int32
 * array [num_seqs][max_blocks_per_seq] and new tokens reach the pool through an int64
 * slot mapping ("vLLM: what PagedAttention turned into", section "The problem
 * PagedAttention was actually solving"). Block id 0 is the null block: an ordinary block
 * that "no block" points at, so that padding needs no sentinel ("vLLM: what
 * PagedAttention turned into", section "The block pool").
 *
 * Layouts (all row-major, all device memory, element type given by pa_dtype):
 *   k_cache, v_cache   [num_blocks][num_kv_heads][16][head_dim]  (one (block, head) page
 *                      of 16 x head_dim elements is contiguous)
 *   slot               physical_block * 16 + offset_in_block; position p of a sequence
 *                      lives in logical block p / 16 at offset p % 16 (0-based)
 *   q, out (decode)    [num_seqs][num_q_heads][head_dim]
 *   q, out (prefill)   [total_query_tokens][num_q_heads][head_dim], sequences packed in
 *                      the order of query_start_loc
 *   GQA                query head h reads kv head h / (num_q_heads / num_kv_heads)
 *
 * Conventions shared by every entry point:
 *   - Every pointer is a device pointer owned and allocated by the caller; the library
 *     allocates no device memory and keeps no per-call state. Pointers must be 16-byte
 *     aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL = legacy
 *     default stream). They never read device data on the host and never synchronise.
 *   - Arguments that the host can check (null pointers, sizes, head ratio, head_dim,
 *     dtype, workspace size, alignment) are checked before anything is launched; a bad
 *     one returns PA_ERR_INVALID_ARG or PA_ERR_UNSUPPORTED and launches nothing.
 *     A failed launch returns PA_ERR_CUDA.
 *   - Device data that the host cannot check (slots, block ids, lengths) is range-checked
 *     by the kernels: an out-of-range slot is not written, an out-of-range block id or a
 *     length beyond max_blocks_per_seq * 16 is not read; each sets a bit in the device
 *     error word (pa_get_device_errors). Kernels never trap.
 *   - seq_lens[i] counts every key of sequence i, the current token(s) included.
 *   - Only the first ceil(seq_lens[i] / 16) entries of block-table row i are read; the
 *     unused tail of a sequence's last block is never read into a result (its contents
 *     may be anything, NaN included), nor is block 0 unless a table names it.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_BLOCK_SIZE 16

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* a host-checkable argument is wrong; nothing launched  */
    PA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. head_dim 96)           */
    PA_ERR_CUDA = 3           /* a CUDA runtime call or launch failed                   */
} pa_status;

typedef enum {
    PA_F32 = 0,               /* fp32 Q/K/V/out, fp32 arithmetic (no TF32)              */
    PA_BF16 = 1               /* bf16 Q/K/V/out, fp32 accumulation                      */
} pa_dtype;

/* Bits of the device error word. */
#define PA_DEVERR_SLOT_RANGE   0x1u  /* reshape_and_cache met a slot >= num_blocks * 16   */
#define PA_DEVERR_BLOCK_RANGE  0x2u  /* a block-table entry outside [0, num_blocks)       */
#define PA_DEVERR_LEN_RANGE    0x4u  /* a length beyond the table row or max_seq_len      */
#define PA_DEVERR_WAIT_TIMEOUT 0x8u  /* a bounded pipeline wait gave up (results invalid) */

/*
 * pa_reshape_and_cache: write the K/V rows of num_tokens new tokens into their slots.
 * For token t with s = slot_mapping[t] >= 0, and every kv head h:
 *   k_cache[s / 16][h][s % 16][:] = k[t][h][:]   and the same for v.
 * The copy is bitwise in the stored type. A negative slot means "no write" (padding may
 * use either a negative slot or a slot inside null block 0). Slots must be distinct
 * unless they point into block 0 (duplicate non-null slots give an unspecified winner).
 *
 *   k, v          [num_tokens][num_kv_heads][head_dim]   (read)
 *   k_cache       [num_blocks][num_kv_heads][16][head_dim] (written at the slots)
 *   slot_mapping  [num_tokens] int64                       (read)
 * Source: "vLLM: what PagedAttention turned into", section "The problem PagedAttention
 * was actually solving" (int64 slot_mapping); "My Understanding of vLLM and
 * PagedAttention", "Step 3 - Tokens Generated Sequentially" (new K/V are added to the
 * cache as tokens are produced).
 */
PA_API pa_status pa_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                               const int64_t* slot_mapping, int32_t num_tokens,
                               int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                               pa_dtype dtype, void* stream);

/*
 * pa_decode_workspace_size: bytes of device scratch that pa_decode needs for this shape on
 * the current device (split-KV partial results and one merge counter per (sequence, kv
 * head)). The caller allocates it and zero-fills it once before its first use; every call
 * that completes without a device error leaves it zero-filled again, so the same buffer
 * serves any number of later calls (and CUDA-graph replays) without re-initialisation.
 * After a call that raised PA_DEVERR_WAIT_TIMEOUT, zero-fill it again. Calls that use the
 * same workspace must not overlap on the GPU.
 */
PA_API size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t max_seq_len, pa_dtype dtype);

/*
 * pa_decode: one query row per sequence, at position seq_lens[i] - 1, attending to keys
 * 0..seq_lens[i]-1 gathered through block_table row i inside the kernel:
 *   out[i][h] = softmax_j(scale * q[i][h] . K_i[j]) V_i[j],  K_i[j] = k_cache[bt[i][j/16]][h/G][j%16]
 * A sequence with seq_lens[i] == 0 gets an all-zero output row.
 * Long sequences are split into pieces whose (max, sum, partial output) are merged with a
 * log-sum-exp reduce: on the bf16 path (GQA groups of 4..16) by the last warp to finish a
 * piece of each (sequence, kv head), inside the same kernel; on the general path by a
 * separate reduce kernel. Everything launches on `stream`.
 *
 *   out            [num_seqs][num_q_heads][head_dim]           (written)
 *   q              [num_seqs][num_q_heads][head_dim]           (read)
 *   block_table    [num_seqs][max_blocks_per_seq] int32         (read)
 *   seq_lens       [num_seqs] int32, each in [0, max_seq_len]   (read)
 *   max_seq_len    host-side upper bound of seq_lens (the host never reads seq_lens)
 *   scale          logit scale, usually 1/sqrt(head_dim)
 *   workspace      >= pa_decode_workspace_size(...) bytes of device scratch, 16-B aligned,
 *                  zero-filled before its first use (see pa_decode_workspace_size)
 * Supported: head_dim 64 or 128; num_q_heads % num_kv_heads == 0; bf16 or fp32.
 * Source: "My Understanding of vLLM and PagedAttention", sections "PagedAttention CUDA
 * Kernel" and "Step 4 - Attention Computation" (gather scattered blocks, restore logical
 * order, compute attention); "vLLM Internals", section 4.1 (block tables read inside the
 * attention kernel).
 */
PA_API pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_table, int32_t max_blocks_per_seq,
                    const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t num_blocks, float scale, pa_dtype dtype,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_prefill_chunk: causal attention for a chunk of new query tokens per sequence, on top
 * of the sequence's earlier context already in the pool (chunked prefill: a long prompt is
 * processed in pieces interleaved with decode, "vLLM Internals", section 2; a chunk is
 * whatever the token budget leaves, "vLLM: what PagedAttention turned into", section "The
 * scheduler"). Chunk rows are bottom-right aligned: sequence i has
 * C_i = query_start_loc[i+1] - query_start_loc[i] query rows; row r sits at position
 * seq_lens[i] - C_i + r and attends to keys 0..seq_lens[i] - C_i + r. The chunk's own K/V
 * must already be in the pool (pa_reshape_and_cache first).
 *
 *   out, q          [query_start_loc[num_seqs]][num_q_heads][head_dim]
 *   block_table     [num_seqs][max_blocks_per_seq] int32
 *   seq_lens        [num_seqs] int32, total keys incl. this chunk, <= max_seq_len
 *   query_start_loc [num_seqs + 1] int32 prefix sums of chunk lengths (starts at 0),
 *                   every chunk length in [0, min(seq_lens[i], max_chunk_len)]
 * Supported: bf16, head_dim 128 (tensor-core path) and the general CUDA-core path for
 * head_dim 64/128 in bf16 or fp32.
 */
PA_API pa_status pa_prefill_chunk(void* out, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_table, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, const int32_t* query_start_loc,
                           int32_t num_seqs, int32_t max_chunk_len, int32_t max_seq_len,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t num_blocks, float scale, pa_dtype dtype, void* stream);

/*
 * pa_decode_noalloc: pa_decode for callers that cannot allocate device memory. The source
 * pages have no counterpart for this entry point; it exists for callers such as a host
 * framework that owns the whole device-memory budget and lets no plug-in allocate, a plug-in
 * that only receives tensors and has no allocator, or a latency-critical path that must not
 * call cudaMalloc/cudaFree (they can synchronise the device).
 *
 * Same arguments and results as pa_decode, without the workspace: the split-KV scratch lives
 * in a fixed array of PA_DECODE_NOALLOC_MAX_BYTES that the library holds in device memory on
 * every GPU that loads it, until the process exits. The call allocates nothing (no
 * cudaMalloc, cudaFree or allocating library routine).
 *   - Shapes whose pa_decode_workspace_size exceeds PA_DECODE_NOALLOC_MAX_BYTES are rejected
 *     with PA_ERR_UNSUPPORTED before anything is launched.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *     with that device current; make that first call before any stream capture.
 *   - Every call shares the one array, which keeps what the previous call left; the call
 *     itself clears the part that must start at zero (an asynchronous memset on `stream`).
 *     Calls that overlap on the GPU (different streams, or concurrent graphs) race on the
 *     array and give wrong results: serialise them.
 */
#define PA_DECODE_NOALLOC_MAX_BYTES (16u * 1024u * 1024u)

PA_API pa_status pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_table, int32_t max_blocks_per_seq,
                                   const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t num_blocks, float scale, pa_dtype dtype, void* stream);

/*
 * pa_get_device_errors: read the device error word of the current device (PA_DEVERR_*
 * bits OR-ed by the kernels since the last clear) into *errors, and clear it when
 * `clear` is non-zero. Synchronises the current device. The library owns the word.
 */
PA_API pa_status pa_get_device_errors(uint32_t* errors, int32_t clear);

/* pa_status_string: static, human-readable name of a status code. */
PA_API const char* pa_status_string(pa_status status);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
