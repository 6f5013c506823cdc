// Chunked prefill: causal attention of a chunk of new query tokens over the sequence's keys in
// the pool ("vLLM Internals", section 2: long prompts are split into chunks interleaved with
// decode; "vLLM: what PagedAttention turned into", "The scheduler": a chunk is what the token
// budget leaves). Chunk rows are bottom-right aligned: row r of a chunk of C tokens of a
// sequence with L keys sits at position L - C + r.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

cudaError_t launch_prefill(const PrefillArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
    (void)dev;
    const int32_t total_rows = a.num_seqs * a.max_chunk_len;  // upper bound; extra rows exit at once
    return launch_prefill_simt(a, total_rows, stream);
}

}  // namespace pa
