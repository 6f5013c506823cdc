// Internal host-side interface between the C ABI (pa_api.cu) and the kernel translation
// units. Not installed; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// Block sizes the kernels accept: powers of two from 16 to 128 tokens. The kernels walk a
// block as block_size / 16 pages of 16 tokens; page j of a sequence is sub-page
// j % (block_size / 16) of logical block j / (block_size / 16).
inline bool block_size_ok(int32_t bs) { return bs == 16 || bs == 32 || bs == 64 || bs == 128; }
inline int block_size_log2(int32_t bs) { return bs == 128 ? 7 : bs == 64 ? 6 : bs == 32 ? 5 : 4; }

// ------------------------------------------------------------------------------------------
// reshape_and_cache
// ------------------------------------------------------------------------------------------
struct ReshapeArgs {
    const void* k;
    const void* v;
    void* k_cache;
    void* v_cache;
    const int64_t* slot_mapping;
    int32_t num_tokens, num_kv_heads, head_dim, num_blocks;
    int32_t elem_bytes;
    int32_t block_size;  // tokens per block: 16, 32, 64 or 128
    uint32_t* err;
};
cudaError_t launch_reshape_and_cache(const ReshapeArgs& a, int num_sms, cudaStream_t stream);

// ------------------------------------------------------------------------------------------
// copy_blocks (copy-on-write pairs of the block manager)
// ------------------------------------------------------------------------------------------
struct CopyBlocksArgs {
    void* k_cache;
    void* v_cache;
    const int32_t* pairs;  // device [num_pairs][2] (src, dst)
    int32_t num_pairs, num_kv_heads, head_dim, num_blocks, elem_bytes;
    int32_t block_size;
    uint32_t* err;
};
cudaError_t launch_copy_blocks(const CopyBlocksArgs& a, cudaStream_t stream);

// ------------------------------------------------------------------------------------------
// decode
// ------------------------------------------------------------------------------------------
// Attention over a part of each row's keys, per row r (= sequence * H_q + q head): the
// normalised output at o + r * D (fp32) and its (max, sum) at ml[r] (log2 domain), so that
// parts over disjoint key ranges merge exactly by the log-sum-exp rule.
struct PartOut {
    float* o = nullptr;
    float2* ml = nullptr;
};

struct DecodeArgs {
    void* out;
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_table;
    int32_t max_blocks_per_seq;
    const int32_t* seq_lens;
    int32_t num_seqs, max_seq_len, num_q_heads, num_kv_heads, head_dim, num_blocks;
    float scale;
    pa_dtype dtype;
    void* workspace;
    size_t workspace_bytes;
    uint32_t* err;
    int32_t block_size;  // tokens per block: 16, 32, 64 or 128
    // append (balanced path only; null otherwise): sequence i's new token at position
    // seq_lens[i] - 1, rows [num_seqs][num_kv_heads][head_dim], written to slot_mapping[i]
    const void* k_new = nullptr;
    const void* v_new = nullptr;
    const int64_t* slot_mapping = nullptr;
    // the kernel before this one on the stream writes neither seq_lens nor block_table
    bool tables_ready = false;
    // ... nor the pool rows this call reads (implies tables_ready)
    bool pool_ready = false;
    // balanced path: keys [len_offset, seq_lens[i]) only (the caller's table rows begin
    // len_offset / block_size entries before block_table; with len_offset > 0 the kernel checks
    // that every row's first entries equal row 0's), and, with part.o set, each row's
    // normalised fp32 output and (max, sum) instead of the bf16 output
    int32_t len_offset = 0;
    PartOut part;
};

// A pipeline wait gives up after this long; the kernel then raises PA_DEVERR_WAIT_TIMEOUT,
// stops issuing copies and runs to completion without writing results.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

// Wait drill (a test hook): with kind != kDrillOff the named kernel announces more bytes on one
// barrier phase than any copy brings, so that one bounded wait runs out; limit_ns then replaces
// the kernels' wait limit. Set through pa_debug_set_wait_drill; read by the launchers.
enum WaitDrillKind : int32_t { kDrillOff = 0, kDrillDecodeStage = 1, kDrillPrefillKTile = 2 };
struct WaitDrill {
    int32_t kind;
    uint64_t limit_ns;
};
WaitDrill wait_drill();

enum DecodePath : int {
    kDecodeSimtSplit = 0,   // CUDA-core kernel over (sequence, kv head, partition) + reduce
    kDecodeMmaBalanced = 1  // persistent TMA + mma.sync kernel over a balanced page list + reduce
};

struct DecodePlan {
    DecodePath path;
    int32_t partition_tokens;  // simt: tokens per partition (multiple of 16)
    int32_t num_partitions;    // simt: ceil(max_seq_len / partition_tokens)
    int32_t head_chunks;       // simt: q heads are processed in chunks of up to 4
    int32_t num_ctas;          // balanced: persistent grid size
    int32_t warps;             // balanced: independent streaming warps per CTA
    int32_t stages;            // balanced: ring stages per warp
    uint32_t stage_bytes;      // balanced: bytes per stage (K page, V page, query rows)
    uint32_t smem_bytes;       // balanced: dynamic shared memory per CTA
    int32_t light_ctas;        // balanced: the last light_ctas CTAs (the last to start) get
    int32_t light_units;       //   light_units pages fewer than the others
    size_t workspace_bytes;
};

struct DeviceInfo {
    int device;
    int num_sms;
    int max_smem_optin;
};

// Fills `info` for the current device (cached per device after the first call).
cudaError_t current_device_info(DeviceInfo* info);

// max_ctas > 0 caps the persistent grid of the balanced path (the SMs it may hold while
// another kernel runs beside it); the workspace never grows with a smaller grid.
// append: the balanced path's stages also carry the appended token's rows.
DecodePlan plan_decode(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                       int32_t max_seq_len, pa_dtype dtype, const DeviceInfo& dev, int32_t max_ctas = 0,
                       bool append = false);
cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream);

// Balanced bf16 path (decode_balanced.cu): fills `plan` and returns true when the shape is
// eligible (GQA group 4..16, head_dim 64/128, at most 1024 sequences) and fits the device.
bool plan_decode_balanced(int32_t num_seqs, int32_t num_kv_heads, int32_t group, int32_t head_dim,
                          const DeviceInfo& dev, DecodePlan* plan, int32_t max_ctas = 0, bool append = false);
cudaError_t launch_decode_balanced(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream);

// Decode over a prefix shared by every sequence (shared_prefix.cu): the suffixes by the
// balanced decode kernel on a grid capped to leave prefix_ctas SMs, written as fp32 parts;
// then the prefix by the tensor-core prefill kernel in shared-prefix mode, launched so that it
// runs beside the decode and merges the suffix parts into the output at its end. Workspace: the
// decode's workspace, then the suffix parts [S][H_q][D] fp32 at parts_o_off and their (max,
// sum) [S][H_q][2] at parts_ml_off.
struct SharedPrefixPlan {
    int32_t prefix_ctas = 0;
    DecodePlan dplan{};
    size_t parts_o_off = 0, parts_ml_off = 0, total = 0;
};
SharedPrefixPlan plan_shared_prefix(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                    int32_t max_seq_len, int32_t prefix_tokens, const DeviceInfo& dev);

// SIMT path (decode_simt.cu).
cudaError_t launch_decode_simt(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream);
int simt_heads_per_cta();

// ------------------------------------------------------------------------------------------
// prefill
// ------------------------------------------------------------------------------------------
// Tensor-core prefill in shared-prefix mode: one query row per decode sequence, all of them
// over the same `len` prefix keys (block-table row 0), no causal bound. Each row's suffix part
// (keys past the prefix, computed by the decode kernel launched just before) is merged in
// before the bf16 output is written; the kernel waits for that decode grid only there.
struct SharedPrefixPart {
    int32_t rows = 0;  // 0: ordinary chunked prefill
    int32_t len = 0;
    const float* suffix_o = nullptr;    // [rows][H_q][D]
    const float2* suffix_ml = nullptr;  // [rows][H_q]
};

struct PrefillArgs {
    void* out;
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_table;
    int32_t max_blocks_per_seq;
    const int32_t* seq_lens;
    const int32_t* query_start_loc;
    int32_t num_seqs, max_chunk_len, max_seq_len, num_q_heads, num_kv_heads, head_dim, num_blocks;
    float scale;
    pa_dtype dtype;
    uint32_t* err;
    int32_t block_size;  // tokens per block: 16, 32, 64 or 128
    SharedPrefixPart sp;  // shared-prefix mode (tensor-core path only) when sp.rows > 0
};
// total_rows: number of chunk rows (query_start_loc[num_seqs]); the host cannot read it, so
// the caller passes an upper bound (grid rows past the end exit at once).
cudaError_t launch_prefill(const PrefillArgs& a, const DeviceInfo& dev, cudaStream_t stream);
// General CUDA-core path (any dtype / head_dim 64/128): one CTA per chunk row and head chunk.
cudaError_t launch_prefill_simt(const PrefillArgs& a, int32_t total_rows, cudaStream_t stream);

// ------------------------------------------------------------------------------------------
// tensor maps (driver entry point resolved at run time; no libcuda link needed)
// ------------------------------------------------------------------------------------------
// Encodes a 2-D bf16 tensor map over `rows` rows of `cols` elements (row pitch cols*2 bytes)
// with a box of box_cols x box_rows and 128-byte swizzle. `map` must point to 128 bytes.
cudaError_t encode_bf16_2d_sw128(void* map, const void* base, uint64_t cols, uint64_t rows,
                                 uint32_t box_cols, uint32_t box_rows);
// 3-D variant: dims (innermost first) d0 x d1 x d2 with byte strides s1 (dim 1) and s2 (dim 2).
cudaError_t encode_bf16_3d_sw128(void* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                                 uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2);

}  // namespace pa
