// K1 reshape_and_cache: scatter the K/V rows of new tokens into their pool slots.
//
// New K and V entries are added to the cache as tokens are produced ("My Understanding of
// vLLM and PagedAttention", "Step 3 - Tokens Generated Sequentially"); the destination of
// token t is the int64 slot slot_mapping[t] = physical_block * block_size + offset ("vLLM:
// what PagedAttention turned into", "The problem PagedAttention was actually solving"; the
// block size is 16 by default, and the same page reports 16 to 128 working alike).
//
// Pure data movement: an item is one 16-byte chunk of a (token, kv head) row of K and the same
// chunk of V. A row of head_dim elements is head_dim*elem/16 chunks (16 for bf16 D128), so a
// warp covers two rows with fully coalesced 16-byte accesses on both sides. Each thread moves
// kUnroll items a grid stride apart, issuing all of their slot and row loads before the first
// store, so that every thread keeps kUnroll x 32 bytes of loads in flight. Loads of the new
// rows are streaming (read once); stores keep the default L2 policy because attention reads
// the new tokens right after.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kUnroll = 4;

__global__ void __launch_bounds__(256) reshape_and_cache_kernel(const int4* __restrict__ k,
                                                                const int4* __restrict__ v,
                                                                int4* __restrict__ k_cache,
                                                                int4* __restrict__ v_cache,
                                                                const int64_t* __restrict__ slot_mapping,
                                                                uint32_t num_items, uint32_t chunks_per_row,
                                                                uint32_t num_kv_heads, int64_t num_slots,
                                                                uint32_t bs_log2, uint32_t* err) {
    // Programmatic launch: wait for the kernel before this one (it may still read the pool or
    // produce k, v and the slots), then let the next kernel's grid be scheduled.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
    for (uint64_t base = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x; base < num_items;
         base += stride * kUnroll) {
        int64_t slot[kUnroll];
        int4 kv[kUnroll], vv[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint64_t i = base + u * stride;
            slot[u] = -1;
            if (i < num_items) {
                const uint32_t t = static_cast<uint32_t>(i) / chunks_per_row / num_kv_heads;  // token (i < 2^31)
                slot[u] = __ldg(slot_mapping + t);
                kv[u] = __ldcs(k + i);
                vv[u] = __ldcs(v + i);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint64_t i = base + u * stride;
            if (i >= num_items || slot[u] < 0) continue;  // past the end, or padding: no write
            if (slot[u] >= num_slots) {                   // outside the pool: never written
                raise_error(err, PA_DEVERR_SLOT_RANGE);
                continue;
            }
            const uint32_t row = static_cast<uint32_t>(i) / chunks_per_row;  // (token, head)
            const uint32_t c = static_cast<uint32_t>(i) - row * chunks_per_row;
            const uint32_t h = row % num_kv_heads;
            const int64_t block = slot[u] >> bs_log2;
            const int64_t offset = slot[u] - (block << bs_log2);
            const int64_t dst = (((block * num_kv_heads + h) << bs_log2) + offset) * chunks_per_row + c;
            k_cache[dst] = kv[u];
            v_cache[dst] = vv[u];
        }
    }
}

}  // namespace

cudaError_t launch_reshape_and_cache(const ReshapeArgs& a, int num_sms, cudaStream_t stream) {
    const int32_t chunks_per_row = a.head_dim * a.elem_bytes / 16;
    const int64_t num_items = static_cast<int64_t>(a.num_tokens) * a.num_kv_heads * chunks_per_row;
    if (num_items == 0) return cudaSuccess;
    if (num_items > 0x7fffffffLL) return cudaErrorInvalidValue;  // host checks this first
    const int threads = 256;
    // kUnroll items per thread; at most what stays resident (8 x 256 threads per SM).
    int64_t blocks = (num_items + threads * kUnroll - 1) / (threads * kUnroll);
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, reshape_and_cache_kernel, static_cast<const int4*>(a.k),
                              static_cast<const int4*>(a.v), static_cast<int4*>(a.k_cache),
                              static_cast<int4*>(a.v_cache), a.slot_mapping, static_cast<uint32_t>(num_items),
                              static_cast<uint32_t>(chunks_per_row), static_cast<uint32_t>(a.num_kv_heads),
                              static_cast<int64_t>(a.num_blocks) * a.block_size,
                              static_cast<uint32_t>(block_size_log2(a.block_size)), a.err);
}

}  // namespace pa
