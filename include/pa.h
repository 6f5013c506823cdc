/*
 * pa.h - C ABI of the GB300 (sm_103a) paged-KV attention library (libpa.so).
 *
 * The KV cache is a pool of fixed-size physical blocks of 16 tokens (or 32, 64 or 128
 * through the *_bs entry points) placed anywhere in device memory; a sequence reaches its blocks through a block table that maps logical
 * block i to a physical block id ("vLLM Internals: From PagedAttention to Removing
 * PagedAttention", section 1.1; "My Understanding of vLLM and PagedAttention", sections
 * "Logical Blocks", "Physical Blocks" and "Block Table"). The table is a dense int32
 * array [num_seqs][max_blocks_per_seq] and new tokens reach the pool through an int64
 * slot mapping ("vLLM: what PagedAttention turned into", section "The problem
 * PagedAttention was actually solving"). Block id 0 is the null block: an ordinary block
 * that "no block" points at, so that padding needs no sentinel ("vLLM: what
 * PagedAttention turned into", section "The block pool").
 *
 * Layouts (all row-major, all device memory, element type given by pa_dtype; BS is the
 * block size, 16 for the plain entry points and the block_size argument of the *_bs ones):
 *   k_cache, v_cache   [num_blocks][num_kv_heads][BS][head_dim]  (one (block, head) page
 *                      of BS x head_dim elements is contiguous)
 *   slot               physical_block * BS + offset_in_block; position p of a sequence
 *                      lives in logical block p / BS at offset p % BS (0-based)
 *   q, out (decode)    [num_seqs][num_q_heads][head_dim]
 *   q, out (prefill)   [total_query_tokens][num_q_heads][head_dim], sequences packed in
 *                      the order of query_start_loc
 *   GQA                query head h reads kv head h / (num_q_heads / num_kv_heads)
 *
 * Conventions shared by every entry point:
 *   - Every pointer is a device pointer owned and allocated by the caller (the block
 *     manager's calls, which take host arrays, excepted); the library allocates no device
 *     memory at run time and keeps no per-call state. Per device it holds the error word, the
 *     fixed scratch of pa_decode_noalloc, and pa_step's side stream and two events. Device
 *     pointers must be 16-byte aligned unless an entry point states otherwise.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL = legacy
 *     default stream). They never read device data on the host and never synchronise
 *     (pa_get_device_errors excepted).
 *   - Arguments that the host can check (null pointers, sizes, head ratio, head_dim,
 *     dtype, workspace size, alignment) are checked before anything is launched; a bad
 *     one returns PA_ERR_INVALID_ARG or PA_ERR_UNSUPPORTED and launches nothing.
 *     A failed launch returns PA_ERR_CUDA.
 *   - Device data that the host cannot check (slots, block ids, lengths) is range-checked
 *     by the kernels: an out-of-range slot is not written, an out-of-range block id or a
 *     length beyond max_blocks_per_seq * BS is not read; each sets a bit in the device
 *     error word (pa_get_device_errors). Kernels never trap.
 *   - seq_lens[i] counts every key of sequence i, the current token(s) included.
 *   - Only the first ceil(seq_lens[i] / BS) entries of block-table row i are read; the
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
    PA_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed                   */
    PA_ERR_NO_SPACE = 4       /* block manager: not enough free blocks (nothing changed),
                                 or an output array too small for the answer            */
} pa_status;

typedef enum {
    PA_F32 = 0,               /* fp32 Q/K/V/out, fp32 arithmetic (no TF32)              */
    PA_BF16 = 1               /* bf16 Q/K/V/out, fp32 accumulation                      */
} pa_dtype;

/* Bits of the device error word. */
#define PA_DEVERR_SLOT_RANGE   0x1u  /* reshape_and_cache met a slot >= num_blocks * BS   */
#define PA_DEVERR_BLOCK_RANGE  0x2u  /* a block-table entry outside [0, num_blocks)       */
#define PA_DEVERR_LEN_RANGE    0x4u  /* a length beyond the table row or max_seq_len      */
#define PA_DEVERR_WAIT_TIMEOUT 0x8u  /* a bounded pipeline wait gave up (results invalid) */
#define PA_DEVERR_APPEND_SLOT  0x10u /* pa_decode_append: slot_mapping[i] is not the slot the
                                        block table gives position seq_lens[i] - 1          */
#define PA_DEVERR_PREFIX_MISMATCH 0x20u /* pa_decode_shared_prefix: a table row does not start
                                           with row 0's prefix blocks (results invalid)   */

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
 * Block-size variants. The page "vLLM: what PagedAttention turned into" (intro table and
 * "The problem PagedAttention was actually solving") gives 16 tokens as the block size and
 * reports sizes from 16 to 128 performing alike. Each *_bs entry point is its plain
 * counterpart with the block size as an argument: block_size must be 16, 32, 64 or 128
 * (another positive value returns PA_ERR_UNSUPPORTED, zero or a negative one
 * PA_ERR_INVALID_ARG), and every "16" of the plain entry point's description (pool layout,
 * slot arithmetic, table reads, length bound) reads block_size. The kernels walk a block
 * as block_size / 16 consecutive 16-token pages, so results are bit-identical to the same
 * keys stored in 16-token blocks. pa_decode_workspace_size does not depend on the block size.
 */
PA_API pa_status pa_reshape_and_cache_bs(const void* k, const void* v, void* k_cache, void* v_cache,
                                         const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t num_blocks, int32_t block_size, pa_dtype dtype,
                                         void* stream);

/*
 * pa_decode_workspace_size: bytes of device scratch that pa_decode needs for this shape on
 * the current device (split-KV partial results; on the bf16 path for groups of 4..16 q heads
 * per kv head, also one merge counter per (sequence, kv head) at its start). The caller
 * allocates it and zero-fills it once before its first use. On that bf16 path every call
 * that completes without a device error puts the counters back to zero, so the same buffer
 * serves any number of later calls (and CUDA-graph replays) without re-initialisation. The
 * general path (fp32, or fewer than 4 q heads per kv head) writes plain partial results over
 * the whole buffer: zero-fill it again before a bf16 grouped call reuses a buffer that the
 * general path used, and after a call that raised PA_DEVERR_WAIT_TIMEOUT. Calls that use the
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
 * pa_decode_shared_prefix: pa_decode for a batch whose sequences all begin with the same
 * prefix_tokens keys in the same physical blocks (the first prefix_tokens / 16 entries of every
 * block-table row equal row 0's). Identical prefixes point at the same physical blocks
 * ("vLLM Internals", section 1.2); this call also computes over them once instead of once per
 * sequence. The result is pa_decode's (same arguments, bf16 only), up to rounding: softmax over
 * a sequence's keys is split into the shared prefix and the sequence's own suffix, each reduced
 * to (normalised output, max, sum), and the two are merged by the log-sum-exp rule.
 *   - The suffix part is the balanced decode kernel over keys [prefix_tokens, seq_lens[i]),
 *     on a grid capped to leave SMs for the prefix part, written as fp32 parts into the
 *     workspace; it also checks the table: a row whose prefix entries differ from row 0's sets
 *     PA_DEVERR_PREFIX_MISMATCH (the results are then invalid). The prefix part runs on the
 *     tensor cores, all sequences' query rows of one kv head together against the prefix's key
 *     tiles (no causal bound), as a programmatic dependent launch: it starts on the free SMs
 *     while the decode streams, waits for the decode grid only at its end, merges each row's
 *     suffix part and writes `out`. Both kernels launch on `stream`.
 *   - prefix_tokens: a positive multiple of 16, at most max_seq_len; every seq_lens[i] must be
 *     at least prefix_tokens (a shorter one sets PA_DEVERR_LEN_RANGE).
 *   - Supported: bf16, head_dim 128, 4, 8 or 16 q heads per kv head, at most 1024 sequences
 *     (PA_ERR_UNSUPPORTED otherwise).
 *   - workspace: >= pa_decode_shared_prefix_workspace_size(...) bytes, 16-byte aligned,
 *     zero-filled before its first use, under the rules of pa_decode_workspace_size (its first
 *     part is the suffix decode's workspace).
 *   - flags: 0, or the promises PA_DECODE_TABLES_READY / PA_DECODE_POOL_READY of
 *     pa_decode_append (below) about the kernel launched just before this call; with
 *     POOL_READY that kernel writes no pool row of keys 0 .. seq_lens[i] - 1. They let the
 *     suffix decode scan the lengths and start its first page copies before its wait.
 *     Other bits: PA_ERR_INVALID_ARG.
 * No counterpart entry point exists on the source pages; they describe the sharing of the
 * blocks, and this computes on that sharing.
 */
PA_API size_t pa_decode_shared_prefix_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                                     int32_t head_dim, int32_t max_seq_len, int32_t prefix_tokens);
PA_API pa_status pa_decode_shared_prefix(void* out, const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_table, int32_t max_blocks_per_seq,
                                         const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                         int32_t num_blocks, float scale, int32_t prefix_tokens, void* workspace,
                                         size_t workspace_bytes, uint32_t flags, void* stream);

/*
 * pa_decode_append: one decode step with its new tokens, in one launch where it can be. For
 * each sequence i the token at position seq_lens[i] - 1 is new: its K and V rows k_new[i],
 * v_new[i] ([num_seqs][num_kv_heads][head_dim]) are written to slot slot_mapping[i] of the
 * pool, exactly as pa_reshape_and_cache_bs writes them, and decode attention runs over keys
 * 0 .. seq_lens[i] - 1 as pa_decode_bs does. New K/V reach the cache as each token is produced
 * ("My Understanding of vLLM and PagedAttention", "Step 3 - Tokens Generated Sequentially");
 * fusing the write into the attention launch is this library's, not the pages'.
 *
 * On the bf16 persistent path (GQA groups 4..16) one kernel does both: attention takes the new
 * rows from k_new / v_new, so it never waits for its own pool writes. Elsewhere the call
 * launches pa_reshape_and_cache's kernel and then the decode kernel. Either way the results
 * equal pa_reshape_and_cache_bs followed by pa_decode_bs when slot_mapping[i] is the slot that
 * block-table row i gives position seq_lens[i] - 1; on the fused path a slot that is not (a
 * negative one included) sets PA_DEVERR_APPEND_SLOT, the write still goes to slot_mapping[i]
 * (skipped if negative) and attention uses the new rows at position seq_lens[i] - 1.
 * Arguments as for pa_decode_bs, plus k_new, v_new (16-byte aligned) and slot_mapping
 * (int64 [num_seqs], 8-byte aligned); workspace as for pa_decode.
 *
 * flags: 0, or an OR of the bits below; any other bit returns PA_ERR_INVALID_ARG. The fused
 * kernel is a programmatic launch: it may start while the kernel launched just before it on
 * `stream` still runs, and it waits for that kernel to complete before it reads what the flags
 * do not declare ready. It lets the next kernel start only after that wait, so every kernel
 * before the previous one has completed when it starts.
 *   PA_DECODE_TABLES_READY: the kernel launched just before this call writes neither seq_lens
 *     nor block_table (they come from host copies or an earlier step). The kernel then scans
 *     the lengths and loads its first block ids before the wait; the pool, the queries, the
 *     new rows, the output and the workspace are touched after it.
 *   PA_DECODE_POOL_READY (implies PA_DECODE_TABLES_READY): in addition, that kernel writes no
 *     pool row this call reads (keys 0 .. seq_lens[i] - 2; this call writes the new rows
 *     itself). In a model's decode step the kernel before attention produces q, k_new and
 *     v_new, never the pool, so the promise holds there. The kernel then also starts its first
 *     page copies before the wait; the queries, the new rows, the output and the workspace are
 *     still touched after it.
 */
#define PA_DECODE_TABLES_READY 1u
#define PA_DECODE_POOL_READY 2u

PA_API pa_status pa_decode_append(void* out, const void* q, const void* k_new, const void* v_new,
                                  const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                  const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                  int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t num_blocks, int32_t block_size, float scale,
                                  pa_dtype dtype, void* workspace, size_t workspace_bytes, uint32_t flags,
                                  void* stream);

/* pa_decode with block_size (see the block-size variants above). */
PA_API pa_status pa_decode_bs(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                              int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t num_blocks, int32_t block_size, float scale, pa_dtype dtype,
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

/* pa_prefill_chunk with block_size (see the block-size variants above). */
PA_API pa_status pa_prefill_chunk_bs(void* out, const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                     const int32_t* query_start_loc, int32_t num_seqs, int32_t max_chunk_len,
                                     int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t num_blocks, int32_t block_size, float scale,
                                     pa_dtype dtype, void* stream);

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
 * pa_step: one whole mixed step of the serving loop in one call: write the step's new K/V
 * into the pool, then chunked-prefill attention for the prefill sequences and decode
 * attention for the decode sequences, with the two attention kernels running side by side.
 * The pages make the per-step work a fixed launch sequence with no host round trip ("vLLM:
 * what PagedAttention turned into", "The scheduler" and the model-runner rewrite: persistent
 * buffers and captured graphs remove per-step CPU work); a step mixes prefill chunks with
 * decode tokens ("vLLM Internals", section 2, chunked prefill).
 *
 * Results are those of the three separate calls (pa_reshape_and_cache_bs, then
 * pa_prefill_chunk_bs and pa_decode_bs on the same pool). Decode is bound by HBM and
 * prefill by the tensor cores, so when both are present and decode takes the bf16
 * persistent path, the decode kernel is given decode_sms SMs and prefill runs on the others
 * at the same time:
 *   stream:  reshape_and_cache -> decode (decode_sms persistent CTAs) -> [join]
 *   side:                     +-> prefill ---------------------------+
 * The side stream and two fork/join events are the library's own, one set per device,
 * created by the first call on that device (make it before any stream capture); the
 * fork/join goes through them under a lock, so pa_step is capturable into a CUDA graph
 * (the side stream joins the capture) and calls from several threads serialise their
 * prefills on the one side stream. Otherwise (no prefill, no decode, or a decode shape that
 * takes the general path) the kernels run one after another on `stream`.
 *
 * A part with zero sequences (or zero new tokens) is skipped and its pointers may be NULL.
 * Every argument is checked as the separate entry point would check it before anything is
 * launched. decode_sms: 0 = 27/64 of the device's SMs (64 of 152, the best split measured for
 * a step of 2 GB of decode KV beside 16 x 512-token prefill chunks); otherwise 1..num_SMs
 * (larger values are clamped). On a capped grid the decode kernel runs 10 warps per CTA.
 * workspace: >= pa_decode_workspace_size(num_decode_seqs, ...) bytes, as for
 * pa_decode. timing_events: NULL, or six cudaEvent_t (each may be NULL) recorded before and
 * after reshape_and_cache, prefill and decode on the stream each kernel runs on, for the
 * caller's profiling; they are recorded as external events, so under stream capture they
 * become event-record nodes of the graph (an event between two kernels stops the later one
 * from launching early).
 */
typedef struct {
    /* the pool and the attention shape shared by every part */
    void* k_cache;
    void* v_cache;
    int32_t num_blocks, block_size;            /* block_size: 16, 32, 64 or 128           */
    int32_t num_q_heads, num_kv_heads, head_dim;
    float scale;
    pa_dtype dtype;
    /* new tokens of the step (pa_reshape_and_cache) */
    const void* k_new;
    const void* v_new;
    const int64_t* slot_mapping;
    int32_t num_new_tokens;
    /* chunked-prefill part (pa_prefill_chunk) */
    void* prefill_out;
    const void* prefill_q;
    const int32_t* prefill_block_table;
    int32_t prefill_max_blocks_per_seq;
    const int32_t* prefill_seq_lens;
    const int32_t* query_start_loc;
    int32_t num_prefill_seqs, max_chunk_len, prefill_max_seq_len;
    /* decode part (pa_decode) */
    void* decode_out;
    const void* decode_q;
    const int32_t* decode_block_table;
    int32_t decode_max_blocks_per_seq;
    const int32_t* decode_seq_lens;
    int32_t num_decode_seqs, decode_max_seq_len;
    void* workspace;
    size_t workspace_bytes;
    /* scheduling */
    int32_t decode_sms;
    void* const* timing_events;
} pa_step_desc;

PA_API pa_status pa_step(const pa_step_desc* step, void* stream);

/*
 * pa_get_device_errors: read the device error word of the current device (PA_DEVERR_*
 * bits OR-ed by the kernels since the last clear) into *errors, and clear it when
 * `clear` is non-zero. Synchronises the current device. The library owns the word.
 */
PA_API pa_status pa_get_device_errors(uint32_t* errors, int32_t clear);

/*
 * pa_debug_set_wait_drill: a test hook for the kernels' bounded waits; the source pages have
 * no counterpart. Every pipeline wait in the tensor-core kernels gives up after a time limit
 * (1 s), raises PA_DEVERR_WAIT_TIMEOUT, lets the copies it already issued land, frees its
 * tensor memory and returns without writing its results. The drill makes one such wait run
 * out on purpose, with nothing in flight that the kernel abandons:
 *   PA_DRILL_OFF              normal operation (limit back to 1 s; limit_ns is ignored)
 *   PA_DRILL_DECODE_STAGE     bf16 grouped decode (pa_decode, pa_decode_append, pa_step):
 *                             the warp that holds the first page of the work list announces
 *                             16 bytes more on its first ring stage than its copies bring
 *   PA_DRILL_PREFILL_K_TILE   tensor-core prefill (pa_prefill_chunk, pa_step): the CTA of the
 *                             first Q-tile pair of kv head 0 of the longest sequence announces
 *                             16 bytes more on its first K tile
 * While a drill is on, limit_ns (1000 .. 10^9) is the wait limit of those kernels. The setting
 * is process-wide and is read when a kernel is launched (a captured graph keeps the values of
 * its capture). After a drilled call the results of that call are invalid and the decode
 * workspace must be zero-filled again before its next use. Returns PA_ERR_INVALID_ARG for an
 * unknown kind or a limit out of range, else PA_OK.
 */
#define PA_DRILL_OFF 0
#define PA_DRILL_DECODE_STAGE 1
#define PA_DRILL_PREFILL_K_TILE 2
PA_API pa_status pa_debug_set_wait_drill(int32_t kind, uint64_t limit_ns);

/*
 * pa_debug_decode_slices: a test hook with no counterpart in the source pages; host only, no
 * device call. The bf16 grouped decode kernel cuts its work list of `units` (sequence, kv head,
 * 16-token page) units into `ctas` contiguous slices, one per CTA, and its last `light_ctas`
 * CTAs (the ones that start last when launches overlap) get `light_units` units fewer than the
 * others, when every slice still gets a unit; otherwise the slices are equal. This writes the
 * first unit of each slice to starts[0..ctas] (starts[ctas] = units) and, if `owners` is not
 * null, the slice that holds unit u to owners[u] for u < units, computed by the same code as
 * the kernel's. Errors: PA_ERR_INVALID_ARG for units outside [0, 2^31), ctas < 1 or a null
 * `starts`. Both arrays belong to the caller.
 */
PA_API pa_status pa_debug_decode_slices(int64_t units, int32_t ctas, int32_t light_ctas, int32_t light_units,
                                        int64_t* starts, int32_t* owners);

/* pa_status_string: static, human-readable name of a status code. */
PA_API const char* pa_status_string(pa_status status);

/*
 * ==========================================================================================
 * Block manager (host side): which physical blocks each request owns
 * ==========================================================================================
 * Host memory only, no device calls; one manager per KV pool; not thread-safe (one caller at
 * a time). It produces the block-table rows and slot mappings the kernels above read.
 *
 * Model ("vLLM: what PagedAttention turned into", "The block pool, and the two tricks in it"
 * and "What a block hash actually is"; "vLLM Internals", section 1.2):
 *   - Block 0 is taken at construction as the null block and never handed out.
 *   - Free blocks sit in one eviction-ordered queue; new blocks come from its front. A freed
 *     block without a hash goes to the front (reused first), one with a hash to the back
 *     (evicted last). A request's blocks are freed tail first.
 *   - A freed block keeps its hash and can still be hit; it leaves the cache only when it is
 *     taken for new content.
 *   - Block hash: SHA-256(parent hash || the block's 16 token ids as int32 little-endian ||
 *     extra key), chained from SHA-256(hash_seed); the extra key is the request's salt, on
 *     the first block only; the cache key is hash || group id 0 (4 bytes, big-endian).
 *   - A new request reuses the longest run of cached full blocks of its prompt (stopping at
 *     the first miss), at most (n_tokens - 1) / 16 of them, so at least one token is left to
 *     compute.
 *   - Blocks are reference counted. pa_bm_fork makes a request that shares every block of its
 *     parent (parallel sampling stores the prompt once); appending into a shared, partly
 *     filled last block first moves the request to a private copy, whose (source,
 *     destination) pair waits in the manager until pa_bm_take_copies hands it to
 *     pa_copy_blocks, which must run before the request's next K/V write.
 *   - A full block is entered into the cache once pa_bm_commit reports its K/V computed.
 * Calls that fail return a status and change nothing.
 */
typedef struct pa_block_manager pa_block_manager;

/* A manager for a pool of num_blocks (>= 2) blocks; enable_caching 0 disables prefix reuse;
 * hash_seed NULL = "paged-kv-none-hash". Free with pa_bm_destroy. */
PA_API pa_status pa_bm_create(int32_t num_blocks, int32_t enable_caching, const char* hash_seed,
                              pa_block_manager** out);
/* The same for blocks of block_size tokens (16, 32, 64 or 128; another positive size returns
 * PA_ERR_UNSUPPORTED): every "16" in the descriptions below reads block_size (hash input,
 * prefix-hit cap, slots). */
PA_API pa_status pa_bm_create_bs(int32_t num_blocks, int32_t block_size, int32_t enable_caching,
                                 const char* hash_seed, pa_block_manager** out);
PA_API void pa_bm_destroy(pa_block_manager* bm);
/* Blocks in the free queue (cached-but-free blocks included); -1 for a NULL manager. */
PA_API int32_t pa_bm_num_free_blocks(const pa_block_manager* bm);

/* A new request with its prompt tokens (host int32[n_tokens], n_tokens >= 1) and optional
 * salt bytes; allocates ceil(n_tokens / 16) blocks, the cached prefix ones shared;
 * *num_cached_tokens = tokens whose K/V is already in the pool (a multiple of 16).
 * PA_ERR_INVALID_ARG for a known req_id; PA_ERR_NO_SPACE when the pool is short. */
PA_API pa_status pa_bm_add_request(pa_block_manager* bm, int64_t req_id, const int32_t* tokens, int32_t n_tokens,
                                   const uint8_t* salt, int32_t salt_len, int32_t* num_cached_tokens);
/* Appends n tokens (e.g. one per decode step), allocating blocks at block boundaries and
 * copying a shared, partly filled last block first (copy-on-write). */
PA_API pa_status pa_bm_append_tokens(pa_block_manager* bm, int64_t req_id, const int32_t* tokens, int32_t n);
/* The first num_computed_tokens tokens of the request have their K/V in the pool: its full
 * blocks among them are hashed and entered into the prefix cache. */
PA_API pa_status pa_bm_commit(pa_block_manager* bm, int64_t req_id, int32_t num_computed_tokens);
/* child_id shares every block (and the tokens) of parent_id. */
PA_API pa_status pa_bm_fork(pa_block_manager* bm, int64_t parent_id, int64_t child_id);
/* Releases the request's blocks, tail first. */
PA_API pa_status pa_bm_free_request(pa_block_manager* bm, int64_t req_id);

/* The request's block-table row: block_ids[i] for i < capacity, padded with the null block;
 * *num_blocks = blocks the request holds (PA_ERR_NO_SPACE if more than capacity). */
PA_API pa_status pa_bm_get_blocks(const pa_block_manager* bm, int64_t req_id, int32_t* block_ids, int32_t capacity,
                                  int32_t* num_blocks);
/* Slots (block * 16 + offset) of positions first_pos .. first_pos + n - 1 of the request,
 * which must lie inside its blocks. */
PA_API pa_status pa_bm_slot_mapping(const pa_block_manager* bm, int64_t req_id, int32_t first_pos, int32_t n,
                                    int64_t* slots);
/* Moves up to capacity pending copy-on-write pairs (oldest first) into src / dst;
 * PA_ERR_NO_SPACE if some remain. */
PA_API pa_status pa_bm_take_copies(pa_block_manager* bm, int32_t* src, int32_t* dst, int32_t capacity,
                                   int32_t* n_copies);
/* Inspection: the free queue from front to back, and one block's reference count and hash. */
PA_API pa_status pa_bm_free_queue(const pa_block_manager* bm, int32_t* order, int32_t capacity, int32_t* n);
PA_API pa_status pa_bm_block_info(const pa_block_manager* bm, int32_t block_id, int32_t* ref_count,
                                  uint8_t* hash32, int32_t* has_hash);
/* Pool size for a memory budget: floor(utilization * free_bytes / per-block bytes over all
 * layers, K and V) ("vLLM: what PagedAttention turned into", "Checking the 96.3%": the pool
 * is sized once from a utilisation fraction of free memory); -1 on a bad argument. */
PA_API int64_t pa_bm_num_blocks_for_memory(size_t free_bytes, double utilization, int32_t num_layers,
                                           int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype);
/* The same for blocks of block_size tokens (16, 32, 64 or 128; -1 otherwise). */
PA_API int64_t pa_bm_num_blocks_for_memory_bs(size_t free_bytes, double utilization, int32_t num_layers,
                                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                              pa_dtype dtype);
/* SHA-256 (FIPS 180-4) of n bytes, as the block hashes use it. */
PA_API pa_status pa_sha256(const uint8_t* data, size_t n, uint8_t* out32);

/*
 * pa_copy_blocks: for each of the n_pairs (src, dst) block-id pairs in block_pairs (device
 * int32 [n_pairs][2]), copy block src of k_cache and of v_cache, every kv head, into block
 * dst (the copy-on-write pairs of the block manager). Pairs must not chain (no dst is another
 * pair's src); src == dst is skipped. Out-of-range ids are not copied and set
 * PA_DEVERR_BLOCK_RANGE. Asynchronous on `stream`.
 */
PA_API pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_pairs, int32_t n_pairs,
                                int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, pa_dtype dtype,
                                void* stream);

/* pa_copy_blocks with block_size (see the block-size variants above). */
PA_API pa_status pa_copy_blocks_bs(void* k_cache, void* v_cache, const int32_t* block_pairs, int32_t n_pairs,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
                                   pa_dtype dtype, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
