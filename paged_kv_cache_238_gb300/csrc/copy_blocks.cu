// copy_blocks: the device half of copy-on-write. When a request forked for parallel sampling
// appends into a partly filled last block that it shares, the block manager moves it to a
// private block ("vLLM Internals", section 1.2: shared prefixes with reference counting and
// copy-on-write; "vLLM: what PagedAttention turned into", "What a block hash actually is",
// last paragraph); this kernel copies the K and V of every kv head of each (src, dst) pair.
//
// Pure data movement: grid x = pair, grid y = 16-byte chunks of a block; each thread moves
// one chunk of K and the same chunk of V, coalesced on both sides (a block's K for all heads
// is H_kv * block_size * head_dim * elem contiguous bytes).
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__global__ void __launch_bounds__(256) copy_blocks_kernel(int4* __restrict__ k_cache, int4* __restrict__ v_cache,
                                                          const int32_t* __restrict__ pairs, uint32_t chunks_per_block,
                                                          int32_t num_blocks, uint32_t* err) {
    const int32_t src = __ldg(pairs + 2 * blockIdx.x), dst = __ldg(pairs + 2 * blockIdx.x + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.y == 0) raise_error(err, PA_DEVERR_BLOCK_RANGE);
        return;
    }
    if (src == dst) return;
    const uint32_t c = blockIdx.y * blockDim.x + threadIdx.x;
    if (c >= chunks_per_block) return;
    const int64_t s = static_cast<int64_t>(src) * chunks_per_block + c;
    const int64_t d = static_cast<int64_t>(dst) * chunks_per_block + c;
    k_cache[d] = __ldg(k_cache + s);
    v_cache[d] = __ldg(v_cache + s);
}

}  // namespace

cudaError_t launch_copy_blocks(const CopyBlocksArgs& a, cudaStream_t stream) {
    if (a.num_pairs == 0) return cudaSuccess;
    const uint32_t chunks = static_cast<uint32_t>(static_cast<int64_t>(a.num_kv_heads) * a.block_size * a.head_dim *
                                                  a.elem_bytes / 16);
    dim3 grid(static_cast<unsigned>(a.num_pairs), (chunks + 255) / 256);
    copy_blocks_kernel<<<grid, 256, 0, stream>>>(static_cast<int4*>(a.k_cache), static_cast<int4*>(a.v_cache),
                                                  a.pairs, chunks, a.num_blocks, a.err);
    return cudaGetLastError();
}

}  // namespace pa
