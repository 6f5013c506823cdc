// C ABI of libpa: host-side argument checks, planning and launches. Every entry point checks
// what the host can check before touching the GPU, launches asynchronously on the caller's
// stream and never synchronises (pa_get_device_errors excepted).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "pa_internal.h"

namespace pa {

// ------------------------------------------------------------------------------------------
// device error word (one per device that loads the library)
// ------------------------------------------------------------------------------------------
static __device__ uint32_t g_device_errors;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceCache {
    bool ready;
    DeviceInfo info;
    uint32_t* err;  // device address of g_device_errors on this device
    // pa_step's fork/join: a non-blocking side stream and two events (no timing), created with
    // the cache entry and kept until the process exits
    cudaStream_t side;
    cudaEvent_t fork, join;
};

DeviceCache g_devices[kMaxDevices];
std::mutex g_mutex;
std::mutex g_step_mutex;  // one fork/join at a time per process

PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;

cudaError_t device_cache(DeviceCache** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceCache& c = g_devices[dev];
    if (!c.ready) {
        DeviceInfo info{};
        info.device = dev;
        e = cudaDeviceGetAttribute(&info.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&info.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        void* err = nullptr;
        e = cudaGetSymbolAddress(&err, g_device_errors);
        if (e != cudaSuccess) return e;
        if (!c.side) {
            e = cudaStreamCreateWithFlags(&c.side, cudaStreamNonBlocking);
            if (e != cudaSuccess) return e;
        }
        if (!c.fork) {
            e = cudaEventCreateWithFlags(&c.fork, cudaEventDisableTiming);
            if (e != cudaSuccess) return e;
        }
        if (!c.join) {
            e = cudaEventCreateWithFlags(&c.join, cudaEventDisableTiming);
            if (e != cudaSuccess) return e;
        }
        c.info = info;
        c.err = static_cast<uint32_t*>(err);
        c.ready = true;
    }
    *out = &c;
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(pa_dtype dt) { return dt == PA_F32 ? 4 : 2; }

bool dtype_ok(pa_dtype dt) { return dt == PA_F32 || dt == PA_BF16; }

// Shared checks of the attention entry points.
pa_status check_attention_shape(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t num_blocks, int32_t max_blocks_per_seq, int32_t max_seq_len,
                                 pa_dtype dtype, int32_t block_size) {
    if (!block_size_ok(block_size)) return block_size > 0 ? PA_ERR_UNSUPPORTED : PA_ERR_INVALID_ARG;
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 ||
        max_seq_len < 0)
        return PA_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return PA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return head_dim > 0 ? PA_ERR_UNSUPPORTED : PA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks_per_seq) * block_size)
        return PA_ERR_INVALID_ARG;
    // Pool rows (block, head, token) are addressed with 32-bit coordinates.
    if (static_cast<int64_t>(num_blocks) * num_kv_heads * block_size > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

}  // namespace

cudaError_t current_device_info(DeviceInfo* info) {
    DeviceCache* c = nullptr;
    cudaError_t e = device_cache(&c);
    if (e == cudaSuccess) *info = c->info;
    return e;
}

static cudaError_t resolve_encoder() {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_encode_tiled) return cudaSuccess;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorNotSupported;
    g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return cudaSuccess;
}

cudaError_t encode_bf16_2d_sw128(void* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                                 uint32_t box_rows) {
    cudaError_t e = resolve_encoder();
    if (e != cudaSuccess) return e;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t elem_strides[2] = {1, 1};
    CUresult r = g_encode_tiled(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                const_cast<void*>(base), dims, strides, box, elem_strides,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_bf16_3d_sw128(void* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                                 uint64_t s1_bytes, uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2) {
    cudaError_t e = resolve_encoder();
    if (e != cudaSuccess) return e;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {s1_bytes, s2_bytes};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    CUresult r = g_encode_tiled(static_cast<CUtensorMap*>(map), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                                const_cast<void*>(base), dims, strides, box, elem_strides,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}


namespace {

// ------------------------------------------------------------------------------------------
// argument checks shared by the single-kernel entry points and pa_step
// ------------------------------------------------------------------------------------------
pa_status prepare_reshape(const void* k, const void* v, void* k_cache, void* v_cache, const int64_t* slot_mapping,
                          int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                          int32_t block_size, pa_dtype dtype, ReshapeArgs* a) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (!block_size_ok(block_size)) return block_size > 0 ? PA_ERR_UNSUPPORTED : PA_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return PA_ERR_INVALID_ARG;
    if ((head_dim * elem_bytes(dtype)) % 16 != 0) return PA_ERR_UNSUPPORTED;
    *a = ReshapeArgs{k, v, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim, num_blocks,
                     elem_bytes(dtype), block_size, nullptr};
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PA_ERR_INVALID_ARG;
    const int64_t items = static_cast<int64_t>(num_tokens) * num_kv_heads * (head_dim * elem_bytes(dtype) / 16);
    if (items > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

// Host checks of a decode call that need no device; plan_checked_decode adds the plan.
pa_status prepare_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                         int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_dim, int32_t num_blocks, int32_t block_size, float scale, pa_dtype dtype,
                         void* workspace, size_t workspace_bytes, DecodeArgs* a) {
    pa_status st = check_attention_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks,
                                         max_blocks_per_seq, max_seq_len, dtype, block_size);
    if (st != PA_OK) return st;
    *a = DecodeArgs{out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                    num_q_heads, num_kv_heads, head_dim, num_blocks, scale, dtype, workspace, workspace_bytes,
                    nullptr, block_size};
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_table || !seq_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

// The decode plan for a checked call (max_ctas > 0 caps the persistent grid) and the check
// of the workspace against it.
pa_status plan_checked_decode(const DecodeArgs& a, const DeviceInfo& info, int32_t max_ctas, DecodePlan* plan,
                              bool append = false) {
    *plan = plan_decode(a.num_seqs, a.num_q_heads, a.num_kv_heads, a.head_dim, a.max_seq_len, a.dtype, info,
                        max_ctas, append);
    if (plan->workspace_bytes > 0 &&
        (!a.workspace || a.workspace_bytes < plan->workspace_bytes || !aligned16(a.workspace)))
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

pa_status prepare_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                          const int32_t* query_start_loc, int32_t num_seqs, int32_t max_chunk_len,
                          int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t num_blocks, int32_t block_size, float scale, pa_dtype dtype, PrefillArgs* a) {
    pa_status st = check_attention_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks,
                                         max_blocks_per_seq, max_seq_len, dtype, block_size);
    if (st != PA_OK) return st;
    if (max_chunk_len < 0 || max_chunk_len > max_seq_len) return PA_ERR_INVALID_ARG;
    *a = PrefillArgs{out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, query_start_loc, num_seqs,
                     max_chunk_len, max_seq_len, num_q_heads, num_kv_heads, head_dim, num_blocks, scale, dtype,
                     nullptr, block_size};
    if (num_seqs == 0 || max_chunk_len == 0) return PA_OK;
    if (static_cast<int64_t>(num_seqs) * max_chunk_len > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    if (!out || !q || !k_cache || !v_cache || !block_table || !seq_lens || !query_start_loc)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(query_start_loc) & 3u))
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

bool prefill_has_work(const PrefillArgs& a) { return a.num_seqs > 0 && a.max_chunk_len > 0; }

std::atomic<int32_t> g_drill_kind{kDrillOff};
std::atomic<uint64_t> g_drill_limit{kWaitLimitNs};

}  // namespace

WaitDrill wait_drill() {
    WaitDrill d;
    d.kind = g_drill_kind.load(std::memory_order_relaxed);
    d.limit_ns = d.kind == kDrillOff ? kWaitLimitNs : g_drill_limit.load(std::memory_order_relaxed);
    return d;
}

}  // namespace pa

using namespace pa;

extern "C" {

PA_API const char* pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_NO_SPACE: return "PA_ERR_NO_SPACE";
    }
    return "PA_UNKNOWN_STATUS";
}

PA_API pa_status pa_reshape_and_cache_bs(const void* k, const void* v, void* k_cache, void* v_cache,
                                         const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t num_blocks, int32_t block_size, pa_dtype dtype,
                                         void* stream) {
    ReshapeArgs a;
    pa_status st = prepare_reshape(k, v, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim,
                                   num_blocks, block_size, dtype, &a);
    if (st != PA_OK || num_tokens == 0) return st;
    DeviceCache* dev = nullptr;
    if (device_cache(&dev) != cudaSuccess) return PA_ERR_CUDA;
    a.err = dev->err;
    return launch_reshape_and_cache(a, dev->info.num_sms, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

PA_API pa_status pa_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                                      const int64_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t num_blocks, pa_dtype dtype, void* stream) {
    return pa_reshape_and_cache_bs(k, v, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim,
                                   num_blocks, PA_BLOCK_SIZE, dtype, stream);
}

PA_API pa_status pa_copy_blocks_bs(void* k_cache, void* v_cache, const int32_t* block_pairs, int32_t n_pairs,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
                                   pa_dtype dtype, void* stream) {
    if (n_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (!block_size_ok(block_size)) return block_size > 0 ? PA_ERR_UNSUPPORTED : PA_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return PA_ERR_INVALID_ARG;
    if ((head_dim * elem_bytes(dtype)) % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (n_pairs == 0) return PA_OK;
    if (n_pairs > 0x7fffffff / 2) return PA_ERR_UNSUPPORTED;
    if (!k_cache || !v_cache || !block_pairs) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache) || (reinterpret_cast<uintptr_t>(block_pairs) & 3u))
        return PA_ERR_INVALID_ARG;
    const int64_t chunks = static_cast<int64_t>(num_kv_heads) * block_size * head_dim * elem_bytes(dtype) / 16;
    if (chunks > 0x7fffffffLL || (chunks + 255) / 256 > 65535) return PA_ERR_UNSUPPORTED;
    DeviceCache* dev = nullptr;
    if (device_cache(&dev) != cudaSuccess) return PA_ERR_CUDA;
    CopyBlocksArgs a{k_cache, v_cache, block_pairs, n_pairs, num_kv_heads, head_dim, num_blocks, elem_bytes(dtype),
                     block_size, dev->err};
    return launch_copy_blocks(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_copy_blocks(void* k_cache, void* v_cache, const int32_t* block_pairs, int32_t n_pairs,
                                int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, pa_dtype dtype,
                                void* stream) {
    return pa_copy_blocks_bs(k_cache, v_cache, block_pairs, n_pairs, num_kv_heads, head_dim, num_blocks,
                             PA_BLOCK_SIZE, dtype, stream);
}

PA_API size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t max_seq_len, pa_dtype dtype) {
    if (check_attention_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, 1, (max_seq_len + 15) / 16 + 1,
                              max_seq_len, dtype, PA_BLOCK_SIZE) != PA_OK)
        return 0;
    DeviceCache* dev = nullptr;
    if (device_cache(&dev) != cudaSuccess) return 0;
    return plan_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len, dtype, dev->info)
        .workspace_bytes;
}

PA_API pa_status pa_decode_append(void* out, const void* q, const void* k_new, const void* v_new,
                                  const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                  const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                  int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t num_blocks, int32_t block_size, float scale,
                                  pa_dtype dtype, void* workspace, size_t workspace_bytes, uint32_t flags,
                                  void* stream) {
    if (flags & ~static_cast<uint32_t>(PA_DECODE_TABLES_READY | PA_DECODE_POOL_READY)) return PA_ERR_INVALID_ARG;
    DecodeArgs a;
    pa_status st = prepare_decode(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, num_seqs,
                                  max_seq_len, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale,
                                  dtype, workspace, workspace_bytes, &a);
    if (st != PA_OK) return st;
    ReshapeArgs ra;
    st = prepare_reshape(k_new, v_new, k_cache, v_cache, slot_mapping, num_seqs, num_kv_heads, head_dim, num_blocks,
                         block_size, dtype, &ra);
    if (st != PA_OK || num_seqs == 0) return st;
    DeviceCache* dev = nullptr;
    if (device_cache(&dev) != cudaSuccess) return PA_ERR_CUDA;
    DecodePlan plan;
    st = plan_checked_decode(a, dev->info, 0, &plan, true);
    if (st != PA_OK) return st;
    a.err = ra.err = dev->err;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (plan.path == kDecodeMmaBalanced) {  // one launch: writes and attention
        a.k_new = k_new;
        a.v_new = v_new;
        a.slot_mapping = slot_mapping;
        a.pool_ready = (flags & PA_DECODE_POOL_READY) != 0;
        a.tables_ready = a.pool_ready || (flags & PA_DECODE_TABLES_READY) != 0;
        return launch_decode(a, plan, s) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }
    if (launch_reshape_and_cache(ra, dev->info.num_sms, s) != cudaSuccess) return PA_ERR_CUDA;
    return launch_decode(a, plan, s) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_decode_bs(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                              int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t num_blocks, int32_t block_size, float scale, pa_dtype dtype,
                              void* workspace, size_t workspace_bytes, void* stream) {
    DecodeArgs a;
    pa_status st = prepare_decode(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, num_seqs,
                                  max_seq_len, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale,
                                  dtype, workspace, workspace_bytes, &a);
    if (st != PA_OK || num_seqs == 0) return st;
    DeviceCache* dev = nullptr;
    if (device_cache(&dev) != cudaSuccess) return PA_ERR_CUDA;
    DecodePlan plan;
    st = plan_checked_decode(a, dev->info, 0, &plan);
    if (st != PA_OK) return st;
    a.err = dev->err;
    return launch_decode(a, plan, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                           int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                           int32_t head_dim, int32_t num_blocks, float scale, pa_dtype dtype, void* workspace,
                           size_t workspace_bytes, void* stream) {
    return pa_decode_bs(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                        num_q_heads, num_kv_heads, head_dim, num_blocks, PA_BLOCK_SIZE, scale, dtype, workspace,
                        workspace_bytes, stream);
}

namespace {
// Host checks of a shared-prefix decode call; fills the decode arguments and the plan.
pa_status prepare_shared_prefix(void* out, const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t num_blocks, float scale, int32_t prefix_tokens,
                                void* workspace, size_t workspace_bytes, DecodeArgs* a) {
    pa_status st = prepare_decode(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, num_seqs,
                                  max_seq_len, num_q_heads, num_kv_heads, head_dim, num_blocks, PA_BLOCK_SIZE, scale,
                                  PA_BF16, workspace, workspace_bytes, a);
    if (st != PA_OK) return st;
    if (prefix_tokens <= 0 || prefix_tokens % PA_BLOCK_SIZE != 0 || prefix_tokens > max_seq_len ||
        prefix_tokens / PA_BLOCK_SIZE > max_blocks_per_seq)
        return PA_ERR_INVALID_ARG;
    const int32_t G = num_q_heads / num_kv_heads;
    if (head_dim != 128 || (G != 4 && G != 8 && G != 16)) return PA_ERR_UNSUPPORTED;
    if (num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

// The plan of a checked shared-prefix call and the check of the workspace against it.
pa_status plan_shared_prefix_checked(const DecodeArgs& a, int32_t prefix_tokens, const DeviceInfo& info,
                                     SharedPrefixPlan* plan) {
    *plan = plan_shared_prefix(a.num_seqs, a.num_q_heads, a.num_kv_heads, a.head_dim, a.max_seq_len, prefix_tokens,
                               info);
    if (a.num_seqs == 0) return PA_OK;
    if (plan->dplan.path != kDecodeMmaBalanced) return PA_ERR_UNSUPPORTED;
    if (!a.workspace || a.workspace_bytes < plan->total || !aligned16(a.workspace)) return PA_ERR_INVALID_ARG;
    return PA_OK;
}
}  // namespace

PA_API size_t pa_decode_shared_prefix_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                                     int32_t head_dim, int32_t max_seq_len, int32_t prefix_tokens) {
    DecodeArgs a;
    const void* fake = reinterpret_cast<const void*>(static_cast<uintptr_t>(0x10000));
    if (prepare_shared_prefix(const_cast<void*>(fake), fake, fake, fake, static_cast<const int32_t*>(fake),
                              (max_seq_len + 15) / 16 + 1, static_cast<const int32_t*>(fake), num_seqs, max_seq_len,
                              num_q_heads, num_kv_heads, head_dim, 1, 1.f, prefix_tokens, const_cast<void*>(fake),
                              ~static_cast<size_t>(0), &a) != PA_OK)
        return 0;
    DeviceCache* dev = nullptr;
    if (device_cache(&dev) != cudaSuccess) return 0;
    SharedPrefixPlan plan;
    if (plan_shared_prefix_checked(a, prefix_tokens, dev->info, &plan) != PA_OK) return 0;
    return plan.total;
}

PA_API pa_status pa_decode_shared_prefix(void* out, const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_table, int32_t max_blocks_per_seq,
                                         const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                         int32_t num_blocks, float scale, int32_t prefix_tokens, void* workspace,
                                         size_t workspace_bytes, uint32_t flags, void* stream) {
    if (flags & ~static_cast<uint32_t>(PA_DECODE_TABLES_READY | PA_DECODE_POOL_READY)) return PA_ERR_INVALID_ARG;
    DecodeArgs a;
    pa_status st = prepare_shared_prefix(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens,
                                         num_seqs, max_seq_len, num_q_heads, num_kv_heads, head_dim, num_blocks,
                                         scale, prefix_tokens, workspace, workspace_bytes, &a);
    if (st != PA_OK || num_seqs == 0) return st;
    DeviceCache* dev = nullptr;
    if (device_cache(&dev) != cudaSuccess) return PA_ERR_CUDA;
    SharedPrefixPlan plan;
    st = plan_shared_prefix_checked(a, prefix_tokens, dev->info, &plan);
    if (st != PA_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    float* parts_o = reinterpret_cast<float*>(ws + plan.parts_o_off);
    float2* parts_ml = reinterpret_cast<float2*>(ws + plan.parts_ml_off);
    // (1) each sequence's suffix, keys [prefix_tokens, len), as fp32 parts, on a capped grid
    a.err = dev->err;
    a.workspace = ws;
    a.workspace_bytes = plan.dplan.workspace_bytes;
    a.block_table = block_table + prefix_tokens / PA_BLOCK_SIZE;
    a.len_offset = prefix_tokens;
    a.max_seq_len = max_seq_len - prefix_tokens;
    a.part.o = parts_o;
    a.part.ml = parts_ml;
    a.pool_ready = (flags & PA_DECODE_POOL_READY) != 0;
    a.tables_ready = a.pool_ready || (flags & PA_DECODE_TABLES_READY) != 0;
    if (launch_decode(a, plan.dplan, s) != cudaSuccess) return PA_ERR_CUDA;
    // (2) the prefix, once per kv head: every sequence's query row over row 0's prefix blocks,
    // merged with its suffix part into the output
    PrefillArgs p{};
    p.out = out;
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_table = block_table;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_seqs = 1;
    p.max_chunk_len = num_seqs;
    p.max_seq_len = prefix_tokens;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.head_dim = head_dim;
    p.num_blocks = num_blocks;
    p.scale = scale;
    p.dtype = PA_BF16;
    p.err = dev->err;
    p.block_size = PA_BLOCK_SIZE;
    p.sp.rows = num_seqs;
    p.sp.len = prefix_tokens;
    p.sp.suffix_o = parts_o;
    p.sp.suffix_ml = parts_ml;
    return launch_prefill(p, dev->info, s) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_prefill_chunk_bs(void* out, const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                     const int32_t* query_start_loc, int32_t num_seqs, int32_t max_chunk_len,
                                     int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t num_blocks, int32_t block_size, float scale,
                                     pa_dtype dtype, void* stream) {
    PrefillArgs a;
    pa_status st = prepare_prefill(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens,
                                   query_start_loc, num_seqs, max_chunk_len, max_seq_len, num_q_heads, num_kv_heads,
                                   head_dim, num_blocks, block_size, scale, dtype, &a);
    if (st != PA_OK || !prefill_has_work(a)) return st;
    DeviceCache* dev = nullptr;
    if (device_cache(&dev) != cudaSuccess) return PA_ERR_CUDA;
    a.err = dev->err;
    return launch_prefill(a, dev->info, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

PA_API pa_status pa_prefill_chunk(void* out, const void* q, const void* k_cache, const void* v_cache,
                                  const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                  const int32_t* query_start_loc, int32_t num_seqs, int32_t max_chunk_len,
                                  int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t num_blocks, float scale, pa_dtype dtype,
                                  void* stream) {
    return pa_prefill_chunk_bs(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, query_start_loc,
                               num_seqs, max_chunk_len, max_seq_len, num_q_heads, num_kv_heads, head_dim, num_blocks,
                               PA_BLOCK_SIZE, scale, dtype, stream);
}

PA_API pa_status pa_step(const pa_step_desc* d, void* stream_ptr) {
    if (!d) return PA_ERR_INVALID_ARG;
    if (d->decode_sms < 0 || d->num_new_tokens < 0 || d->num_prefill_seqs < 0 || d->num_decode_seqs < 0)
        return PA_ERR_INVALID_ARG;
    // Each part with work is checked as its own entry point would check it; parts without work
    // are skipped whole (their pointers and sizes may be zero).
    const bool has_new = d->num_new_tokens > 0, has_dec = d->num_decode_seqs > 0;
    ReshapeArgs ra{};
    PrefillArgs pa_{};
    DecodeArgs da{};
    pa_status st = PA_OK;
    if (has_new) {
        st = prepare_reshape(d->k_new, d->v_new, d->k_cache, d->v_cache, d->slot_mapping, d->num_new_tokens,
                             d->num_kv_heads, d->head_dim, d->num_blocks, d->block_size, d->dtype, &ra);
        if (st != PA_OK) return st;
    }
    if (d->num_prefill_seqs > 0) {
        st = prepare_prefill(d->prefill_out, d->prefill_q, d->k_cache, d->v_cache, d->prefill_block_table,
                             d->prefill_max_blocks_per_seq, d->prefill_seq_lens, d->query_start_loc,
                             d->num_prefill_seqs, d->max_chunk_len, d->prefill_max_seq_len, d->num_q_heads,
                             d->num_kv_heads, d->head_dim, d->num_blocks, d->block_size, d->scale, d->dtype, &pa_);
        if (st != PA_OK) return st;
    }
    if (has_dec) {
        st = prepare_decode(d->decode_out, d->decode_q, d->k_cache, d->v_cache, d->decode_block_table,
                            d->decode_max_blocks_per_seq, d->decode_seq_lens, d->num_decode_seqs,
                            d->decode_max_seq_len, d->num_q_heads, d->num_kv_heads, d->head_dim, d->num_blocks,
                            d->block_size, d->scale, d->dtype, d->workspace, d->workspace_bytes, &da);
        if (st != PA_OK) return st;
    }
    const bool has_pre = d->num_prefill_seqs > 0 && prefill_has_work(pa_);
    if (!has_new && !has_pre && !has_dec) return PA_OK;
    DeviceCache* dev = nullptr;
    if (device_cache(&dev) != cudaSuccess) return PA_ERR_CUDA;
    DecodePlan plan{};
    if (has_dec) {
        const int32_t n = dev->info.num_sms;
        const int32_t dflt = (n * 27) / 64 > 0 ? (n * 27) / 64 : 1;  // 64 of 152 SMs
        const int32_t sms = d->decode_sms == 0 ? dflt : (d->decode_sms < n ? d->decode_sms : n);
        st = plan_checked_decode(da, dev->info, has_pre ? sms : 0, &plan);
        if (st != PA_OK) return st;
    }
    ra.err = pa_.err = da.err = dev->err;
    cudaStream_t s = static_cast<cudaStream_t>(stream_ptr);
    void* const* ev = d->timing_events;
    // The caller's timing events become event-record nodes when the stream is being captured
    // (the external flag is valid only under capture).
    auto mark = [&](int i, cudaStream_t on) -> bool {
        if (!ev || !ev[i]) return true;
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(on, &cs) != cudaSuccess) return false;
        const unsigned flags = cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : cudaEventRecordDefault;
        return cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev[i]), on, flags) == cudaSuccess;
    };
    if (has_new) {
        if (!mark(0, s) || launch_reshape_and_cache(ra, dev->info.num_sms, s) != cudaSuccess || !mark(1, s))
            return PA_ERR_CUDA;
    }
    const bool side_by_side = has_pre && has_dec && plan.path == kDecodeMmaBalanced;
    if (!side_by_side) {
        if (has_pre && (!mark(2, s) || launch_prefill(pa_, dev->info, s) != cudaSuccess || !mark(3, s)))
            return PA_ERR_CUDA;
        if (has_dec && (!mark(4, s) || launch_decode(da, plan, s) != cudaSuccess || !mark(5, s)))
            return PA_ERR_CUDA;
        return PA_OK;
    }
    // Fork: the side stream waits for the new tokens; the decode grid is launched first so its
    // persistent CTAs take their SMs before the prefill grid fills the rest.
    std::lock_guard<std::mutex> lock(g_step_mutex);
    if (cudaEventRecord(dev->fork, s) != cudaSuccess) return PA_ERR_CUDA;
    if (!mark(4, s) || launch_decode(da, plan, s) != cudaSuccess || !mark(5, s)) return PA_ERR_CUDA;
    if (cudaStreamWaitEvent(dev->side, dev->fork, 0) != cudaSuccess) return PA_ERR_CUDA;
    if (!mark(2, dev->side) || launch_prefill(pa_, dev->info, dev->side) != cudaSuccess || !mark(3, dev->side))
        return PA_ERR_CUDA;
    // Join: later work on `stream` waits for the prefill too.
    if (cudaEventRecord(dev->join, dev->side) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaStreamWaitEvent(s, dev->join, 0) != cudaSuccess) return PA_ERR_CUDA;
    return PA_OK;
}

PA_API pa_status pa_debug_set_wait_drill(int32_t kind, uint64_t limit_ns) {
    if (kind == PA_DRILL_OFF) {
        g_drill_kind.store(kDrillOff);
        g_drill_limit.store(kWaitLimitNs);
        return PA_OK;
    }
    if (kind != PA_DRILL_DECODE_STAGE && kind != PA_DRILL_PREFILL_K_TILE) return PA_ERR_INVALID_ARG;
    if (limit_ns < 1000 || limit_ns > kWaitLimitNs) return PA_ERR_INVALID_ARG;
    g_drill_limit.store(limit_ns);
    g_drill_kind.store(kind == PA_DRILL_DECODE_STAGE ? kDrillDecodeStage : kDrillPrefillKTile);
    return PA_OK;
}

PA_API pa_status pa_get_device_errors(uint32_t* errors, int32_t clear) {
    if (!errors) return PA_ERR_INVALID_ARG;
    DeviceCache* dev = nullptr;
    if (device_cache(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpy(&v, dev->err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return PA_ERR_CUDA;
    *errors = v;
    if (clear && cudaMemset(dev->err, 0, sizeof(uint32_t)) != cudaSuccess) return PA_ERR_CUDA;
    return PA_OK;
}

}  // extern "C"
