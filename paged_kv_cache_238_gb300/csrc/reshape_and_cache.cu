// K1 reshape_and_cache: scatter the K/V rows of new tokens into their pool slots.
//
// New K and V entries are added to the cache as tokens are produced ("My Understanding of
// vLLM and PagedAttention", "Step 3 - Tokens Generated Sequentially"); the destination of
// token t is the int64 slot slot_mapping[t] = physical_block * block_size + offset ("vLLM:
// what PagedAttention turned into", "The problem PagedAttention was actually solving"; the
// block size is 16 by default, and the same page reports 16 to 128 working alike).
//
// Pure data movement: each thread moves one 16-byte chunk of a (token, kv head) row of K and
// the same chunk of V. Loads of the new rows are streaming (read once); stores keep the
// default L2 policy because attention reads the new tokens right after. A row of head_dim
// elements is head_dim*elem/16 chunks (16 for bf16 D128), so a warp covers two rows with
// fully coalesced 16-byte accesses on both sides.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

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
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < num_items; i += stride) {
        const uint32_t row = i / chunks_per_row;          // (token, head)
        const uint32_t c = i - row * chunks_per_row;
        const uint32_t t = row / num_kv_heads;
        const uint32_t h = row - t * num_kv_heads;
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;                           // padding: no write
        if (slot >= num_slots) {                          // outside the pool: never written
            raise_error(err, PA_DEVERR_SLOT_RANGE);
            continue;
        }
        const int64_t block = slot >> bs_log2;
        const int64_t offset = slot - (block << bs_log2);
        const int64_t dst = (((block * num_kv_heads + h) << bs_log2) + offset) * chunks_per_row + c;
        const int4 kv = __ldcs(k + i);
        const int4 vv = __ldcs(v + i);
        k_cache[dst] = kv;
        v_cache[dst] = vv;
    }
}

}  // namespace

cudaError_t launch_reshape_and_cache(const ReshapeArgs& a, int num_sms, cudaStream_t stream) {
    const int32_t chunks_per_row = a.head_dim * a.elem_bytes / 16;
    const int64_t num_items = static_cast<int64_t>(a.num_tokens) * a.num_kv_heads * chunks_per_row;
    if (num_items == 0) return cudaSuccess;
    if (num_items > 0x7fffffffLL) return cudaErrorInvalidValue;  // host checks this first
    const int threads = 256;
    // Enough CTAs to keep every SM busy (8 resident x 256 threads), never more than the work.
    int64_t blocks = (num_items + threads - 1) / threads;
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
