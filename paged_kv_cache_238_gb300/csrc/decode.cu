// Decode planning and dispatch: picks the kernel family for a shape and sizes its workspace.
//
//  * bf16 with 4..16 q heads per kv head (head_dim 64/128, up to 1024 sequences): the balanced
//    persistent TMA + mma.sync kernel (decode_balanced.cu). Its work split is derived on the
//    device from seq_lens, so the host needs no length information beyond max_seq_len.
//  * everything else (fp32, small or large groups): the SIMT split-KV kernel (decode_simt.cu),
//    whose partitions are sized here from max_seq_len so that (sequence, kv head, head chunk,
//    partition) items fill the GPU about twice.
#include "pa_internal.h"

namespace pa {

DecodePlan plan_decode(int32_t S, int32_t Hq, int32_t Hkv, int32_t D, int32_t max_seq_len, pa_dtype dt,
                       const DeviceInfo& dev, int32_t max_ctas, bool append) {
    DecodePlan plan{};
    const int32_t G = Hq / Hkv;
    if (dt == PA_BF16 && plan_decode_balanced(S, Hkv, G, D, dev, &plan, max_ctas, append)) return plan;

    plan.path = kDecodeSimtSplit;
    const int32_t heads = simt_heads_per_cta();
    plan.head_chunks = (G + heads - 1) / heads;
    const int64_t items = static_cast<int64_t>(S) * Hkv * plan.head_chunks;
    const int64_t target = 2LL * dev.num_sms;
    int32_t parts = 1;
    if (items < target && max_seq_len > 64) {
        parts = static_cast<int32_t>((target + items - 1) / items);
        parts = parts < (max_seq_len + 63) / 64 ? parts : (max_seq_len + 63) / 64;
    }
    int32_t pt = (max_seq_len + parts - 1) / parts;
    pt = ((pt + 15) / 16) * 16;
    if (pt < 16) pt = 16;
    plan.partition_tokens = pt;
    plan.num_partitions = (max_seq_len + pt - 1) / pt;
    if (plan.num_partitions < 1) plan.num_partitions = 1;
    plan.workspace_bytes = plan.num_partitions > 1
                               ? static_cast<size_t>(S) * Hq * plan.num_partitions * (D + 2) * sizeof(float)
                               : 0;
    return plan;
}

cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    if (a.num_seqs == 0) return cudaSuccess;
    if (plan.path == kDecodeMmaBalanced) return launch_decode_balanced(a, plan, stream);
    return launch_decode_simt(a, plan, stream);
}

}  // namespace pa
