// C ABI of libpa: host-side argument checks, planning and launches. Every entry point checks
// what the host can check before touching the GPU, launches asynchronously on the caller's
// stream and never synchronises (pa_get_device_errors excepted).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

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
};

DeviceCache g_devices[kMaxDevices];
std::mutex g_mutex;

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
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
    if (!block_size_ok(block_size)) return block_size > 0 ? PA_ERR_UNSUPPORTED : PA_ERR_INVALID_ARG;
    if (!dtype_ok(dtype)) return PA_ERR_INVALID_ARG;
    if ((head_dim * elem_bytes(dtype)) % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PA_ERR_INVALID_ARG;
    const int64_t items = static_cast<int64_t>(num_tokens) * num_kv_heads * (head_dim * elem_bytes(dtype) / 16);
    if (items > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    DeviceCache* dev = nullptr;
    if (device_cache(&dev) != cudaSuccess) return PA_ERR_CUDA;
    ReshapeArgs a{k, v, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim, num_blocks,
                  elem_bytes(dtype), block_size, dev->err};
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

PA_API pa_status pa_decode_bs(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                              int32_t num_seqs, int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t num_blocks, int32_t block_size, float scale, pa_dtype dtype,
                              void* workspace, size_t workspace_bytes, void* stream) {
    pa_status st = check_attention_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks,
                                         max_blocks_per_seq, max_seq_len, dtype, block_size);
    if (st != PA_OK) return st;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_table || !seq_lens) return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return PA_ERR_INVALID_ARG;
    DeviceCache* dev = nullptr;
    if (device_cache(&dev) != cudaSuccess) return PA_ERR_CUDA;
    const DecodePlan plan = plan_decode(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len, dtype, dev->info);
    if (plan.workspace_bytes > 0 && (!workspace || workspace_bytes < plan.workspace_bytes || !aligned16(workspace)))
        return PA_ERR_INVALID_ARG;
    DecodeArgs a{out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                 num_q_heads, num_kv_heads, head_dim, num_blocks, scale, dtype, workspace, workspace_bytes,
                 dev->err, block_size};
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

PA_API pa_status pa_prefill_chunk_bs(void* out, const void* q, const void* k_cache, const void* v_cache,
                                     const int32_t* block_table, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                     const int32_t* query_start_loc, int32_t num_seqs, int32_t max_chunk_len,
                                     int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t num_blocks, int32_t block_size, float scale,
                                     pa_dtype dtype, void* stream) {
    pa_status st = check_attention_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks,
                                         max_blocks_per_seq, max_seq_len, dtype, block_size);
    if (st != PA_OK) return st;
    if (max_chunk_len < 0 || max_chunk_len > max_seq_len) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 || max_chunk_len == 0) return PA_OK;
    if (static_cast<int64_t>(num_seqs) * max_chunk_len > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
    if (!out || !q || !k_cache || !v_cache || !block_table || !seq_lens || !query_start_loc)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(query_start_loc) & 3u))
        return PA_ERR_INVALID_ARG;
    DeviceCache* dev = nullptr;
    if (device_cache(&dev) != cudaSuccess) return PA_ERR_CUDA;
    PrefillArgs a{out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, query_start_loc, num_seqs,
                  max_chunk_len, max_seq_len, num_q_heads, num_kv_heads, head_dim, num_blocks, scale, dtype,
                  dev->err, block_size};
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
