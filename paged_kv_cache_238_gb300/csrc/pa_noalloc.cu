// pa_decode_noalloc: pa_decode for callers that cannot allocate device memory.
//
// Some callers cannot hand the library a freshly allocated workspace: a host framework that
// owns the whole device-memory budget and does not let plug-ins allocate, a plug-in that only
// receives tensors from its host and has no allocator of its own, or a latency-critical path
// that must not call cudaMalloc/cudaFree because those calls can synchronise the device. For
// them this entry point runs the same decode kernels with their scratch in a fixed array that
// the library itself holds in device memory (file-scope, one per GPU that loads the library,
// kept until the process exits). Nothing is allocated per call.
#include <cuda_runtime.h>

#include <mutex>

#include "pa_internal.h"

namespace pa {
namespace {

// The fixed scratch. In host code `g_noalloc_scratch` only names a host-side stand-in for the
// symbol; its device address comes from cudaGetSymbolAddress (below) and is what the kernels
// receive.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_DECODE_NOALLOC_MAX_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices];  // device address of the scratch, per device (set up once)

// Resolves the scratch's device address for the current device on the first call there.
cudaError_t noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (p == nullptr) return cudaErrorInvalidSymbol;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" PA_API pa_status pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                                              const int32_t* block_table, int32_t max_blocks_per_seq,
                                              const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                              int32_t num_blocks, float scale, pa_dtype dtype, void* stream) {
    // Shape checks first (no GPU work), exactly as pa_decode would do them.
    const size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len, dtype);
    if (num_seqs > 0 && need == 0) {
        // Either an invalid shape or a shape that needs no scratch: let pa_decode decide.
        void* none = nullptr;
        return pa_decode(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                         num_q_heads, num_kv_heads, head_dim, num_blocks, scale, dtype, none, 0, stream);
    }
    if (need > PA_DECODE_NOALLOC_MAX_BYTES) return PA_ERR_UNSUPPORTED;  // beyond the fixed scratch
    void* scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) return PA_ERR_CUDA;
    // The array keeps whatever the previous call (of any shape or path) left in it; the
    // decode kernels need the leading merge counters at zero, so clear exactly that prefix
    // (one per (sequence, kv head), rounded up to 256 bytes) on the caller's stream.
    if (num_seqs > 0) {
        const size_t counters = ((static_cast<size_t>(num_seqs) * num_kv_heads * 4) + 255) & ~static_cast<size_t>(255);
        const size_t clear = counters < need ? counters : need;
        if (cudaMemsetAsync(scratch, 0, clear, static_cast<cudaStream_t>(stream)) != cudaSuccess) return PA_ERR_CUDA;
    }
    return pa_decode(out, q, k_cache, v_cache, block_table, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
                     num_q_heads, num_kv_heads, head_dim, num_blocks, scale, dtype, scratch,
                     static_cast<size_t>(PA_DECODE_NOALLOC_MAX_BYTES), stream);
}
