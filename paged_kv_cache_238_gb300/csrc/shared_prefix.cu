// Decode over a prefix that every sequence of the batch shares (the same physical blocks in the
// first entries of every block-table row): "vLLM Internals", section 1.2, has identical prefixes
// point at the same physical blocks; this path also computes over them once.
//
// softmax over a sequence's keys splits exactly into parts over disjoint key ranges, each kept
// as (normalised output o_p, max m_p, sum l_p) and merged by the log-sum-exp rule
//   M = max_p m_p,  w_p = l_p 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p.
// The parts here: each sequence's own suffix, attended by the balanced decode kernel over keys
// [prefix, len) and written as fp32 parts, and the shared prefix, attended once per kv head by
// the tensor-core prefill kernel with every sequence's query rows as the rows of one tile set (no
// causal bound). Decode runs first on a grid capped to leave the prefix kernel's CTAs their
// SMs; the prefix kernel is a programmatic dependent that starts at once on those SMs, computes
// its part while decode streams, and waits for the decode grid only before it merges each row's
// suffix part into the output. This file holds the plan.
#include "pa_internal.h"

namespace pa {

SharedPrefixPlan plan_shared_prefix(int32_t S, int32_t Hq, int32_t Hkv, int32_t D, int32_t max_seq_len,
                                    int32_t prefix_tokens, const DeviceInfo& dev) {
    SharedPrefixPlan p;
    (void)prefix_tokens;
    const int32_t G = Hq / Hkv;
    const int32_t q_tiles = (S * G + 127) / 128;  // one per prefix CTA
    p.prefix_ctas = q_tiles * Hkv;
    // decode on the SMs the prefix CTAs leave (at least half of them; more prefix CTAs than
    // that queue behind the decode grid)
    int32_t decode_ctas = dev.num_sms - p.prefix_ctas;
    if (decode_ctas < dev.num_sms / 2) decode_ctas = dev.num_sms / 2;
    const int32_t suffix = max_seq_len - prefix_tokens > 0 ? max_seq_len - prefix_tokens : 1;
    p.dplan = plan_decode(S, Hq, Hkv, D, suffix, PA_BF16, dev, decode_ctas);
    const auto align = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t rows = static_cast<size_t>(S) * Hq;
    p.parts_o_off = align(p.dplan.workspace_bytes);
    p.parts_ml_off = p.parts_o_off + align(rows * D * 4);
    p.total = p.parts_ml_off + align(rows * 8);
    return p;
}

}  // namespace pa
