// SIMT split-KV decode kernel (CUDA cores, fp32 arithmetic) and its log-sum-exp reduce.
//
// Used for fp32 data and for bf16 GQA groups outside 4..16; it also serves as the general
// chunked-prefill path, because a chunk row at position p is exactly a decode query whose
// visible length is p + 1 on the same block-table row. Grid: (query row, kv head x chunk of
// up to 4 q heads, key partition). Each CTA walks its partition's 16-token pages through the
// block table, four warps taking pages round-robin; lanes hold head_dim/32 elements, dot
// products reduce with warp shuffles, the online softmax runs per warp, and the four warps
// merge in shared memory. A sequence split over several partitions writes (m, l, o) per
// partition to the workspace and the reduce kernel merges them:
//   M = max_p m_p,  w_p = l_p 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p   (log2 domain).
#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ==========================================================================================
// SIMT split kernel
// ==========================================================================================
constexpr int kSimtHeads = 4;     // q heads per CTA
constexpr int kSimtThreads = 128;

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<uint16_t>(uint16_t x) { return bf16_bits_to_float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ uint16_t from_f32<uint16_t>(float x) {
    __nv_bfloat16 b = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&b);
}

// Effective length of sequence s: clamped to what the table row can address.
__device__ __forceinline__ int32_t clamped_len(const int32_t* lens, int32_t s, int32_t cap, uint32_t* err) {
    int32_t len = __ldg(lens + s);
    if (len < 0 || len > cap) {
        raise_error(err, PA_DEVERR_LEN_RANGE);
        len = len < 0 ? 0 : cap;
    }
    return len;
}

template <typename T, int D>
__global__ void __launch_bounds__(kSimtThreads) decode_simt_kernel(
    T* __restrict__ out, const T* __restrict__ q, const T* __restrict__ k_cache, const T* __restrict__ v_cache,
    const int32_t* __restrict__ block_table, int32_t max_blocks, const int32_t* __restrict__ seq_lens,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t num_blocks, float scale_log2, int32_t part_tokens,
    int32_t num_parts, int32_t head_chunks, float* __restrict__ ws_o, float* __restrict__ ws_ml,
    const int32_t* __restrict__ query_start_loc, int32_t num_seqs, int32_t sub_log2, uint32_t* err) {
    constexpr int E = D / 32;  // elements per lane
    const int32_t cap_tokens = table_tokens(max_blocks, sub_log2);
    const int32_t row = blockIdx.x;  // query row: a sequence (decode) or a chunk token (prefill)
    const int32_t hk = blockIdx.y / head_chunks;
    const int32_t g0 = (blockIdx.y % head_chunks) * kSimtHeads;
    const int32_t p = blockIdx.z;    // partition of the keys
    const int32_t G = num_q_heads / num_kv_heads;
    const int32_t ng = min(kSimtHeads, G - g0);
    const int32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int32_t s = row, len;
    if (query_start_loc == nullptr) {
        len = clamped_len(seq_lens, s, min(cap_tokens, num_parts * part_tokens), err);
    } else {
        // prefill: chunk row r of sequence s sits at position seq_len - C + r and sees keys
        // 0..position, i.e. a query of visible length seq_len - C + r + 1
        if (row >= __ldg(query_start_loc + num_seqs)) return;  // past the last chunk row
        int32_t lo = 0, hi = num_seqs;
        while (hi - lo > 1) {
            const int32_t mid = (lo + hi) >> 1;
            if (__ldg(query_start_loc + mid) <= row) lo = mid; else hi = mid;
        }
        s = lo;
        const int32_t q0 = __ldg(query_start_loc + s), chunk = __ldg(query_start_loc + s + 1) - q0;
        const int32_t total = clamped_len(seq_lens, s, min(cap_tokens, num_parts * part_tokens), err);
        len = total - chunk + (row - q0) + 1;
        if (len < 1 || chunk > total) {
            raise_error(err, PA_DEVERR_LEN_RANGE);
            len = 0;
        }
    }
    const int32_t parts = (len + part_tokens - 1) / part_tokens;
    if (len == 0) {
        if (p == 0) {
            for (int32_t i = threadIdx.x; i < ng * D; i += kSimtThreads) {
                const int32_t hq = hk * G + g0 + i / D;
                out[(static_cast<int64_t>(row) * num_q_heads + hq) * D + i % D] = from_f32<T>(0.f);
            }
        }
        return;
    }
    if (p >= parts) return;
    const int32_t t0 = p * part_tokens;
    const int32_t t1 = min(len, t0 + part_tokens);

    // q (pre-scaled by scale*log2e) for the CTA's heads, this lane's E elements
    float qv[kSimtHeads][E];
#pragma unroll
    for (int g = 0; g < kSimtHeads; ++g) {
        const int32_t hq = hk * G + g0 + min(g, ng - 1);
        const T* qp = q + (static_cast<int64_t>(row) * num_q_heads + hq) * D + lane * E;
#pragma unroll
        for (int e = 0; e < E; ++e) qv[g][e] = to_f32<T>(qp[e]) * scale_log2;
    }
    float m[kSimtHeads], l[kSimtHeads], acc[kSimtHeads][E];
#pragma unroll
    for (int g = 0; g < kSimtHeads; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) acc[g][e] = 0.f;
    }

    for (int32_t page = t0 / kPageTokens + warp; page * kPageTokens < t1; page += kSimtThreads / 32) {
        const int32_t phys = __ldg(block_table + static_cast<int64_t>(s) * max_blocks + (page >> sub_log2));
        if (phys < 0 || phys >= num_blocks) {
            raise_error(err, PA_DEVERR_BLOCK_RANGE);
            continue;
        }
        const int32_t ntok = min(kPageTokens, t1 - page * kPageTokens);
        const int64_t base =
            ((((static_cast<int64_t>(phys) * num_kv_heads + hk) << sub_log2) + (page & ((1 << sub_log2) - 1))) *
             kPageTokens) * D + lane * E;
        for (int32_t j = 0; j < ntok; ++j) {
            float kr[E], vr[E];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                kr[e] = to_f32<T>(k_cache[base + j * D + e]);
                vr[e] = to_f32<T>(v_cache[base + j * D + e]);
            }
            float sc[kSimtHeads];
#pragma unroll
            for (int g = 0; g < kSimtHeads; ++g) {
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) d = fmaf(qv[g][e], kr[e], d);
                sc[g] = d;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
                for (int g = 0; g < kSimtHeads; ++g) sc[g] += __shfl_xor_sync(0xffffffffu, sc[g], off);
            }
#pragma unroll
            for (int g = 0; g < kSimtHeads; ++g) {
                const float mn = fmaxf(m[g], sc[g]);
                const float corr = exp2f(m[g] - mn);
                const float pj = exp2f(sc[g] - mn);
                l[g] = l[g] * corr + pj;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[g][e] = fmaf(pj, vr[e], acc[g][e] * corr);
                m[g] = mn;
            }
        }
    }

    // merge the four warps
    __shared__ float sm_acc[kSimtThreads / 32][kSimtHeads][D];
    __shared__ float sm_m[kSimtThreads / 32][kSimtHeads], sm_l[kSimtThreads / 32][kSimtHeads];
#pragma unroll
    for (int g = 0; g < kSimtHeads; ++g) {
#pragma unroll
        for (int e = 0; e < E; ++e) sm_acc[warp][g][lane * E + e] = acc[g][e];
        if (lane == 0) {
            sm_m[warp][g] = m[g];
            sm_l[warp][g] = l[g];
        }
    }
    __syncthreads();
    for (int32_t i = threadIdx.x; i < ng * D; i += kSimtThreads) {
        const int32_t g = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kSimtThreads / 32; ++w) M = fmaxf(M, sm_m[w][g]);
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < kSimtThreads / 32; ++w) {
            const float f = exp2f(sm_m[w][g] - M);  // warps without keys: m = -inf -> 0
            num = fmaf(sm_acc[w][g][d], f, num);
            den = fmaf(sm_l[w][g], f, den);
        }
        const int32_t hq = hk * G + g0 + g;
        if (parts == 1) {
            out[(static_cast<int64_t>(row) * num_q_heads + hq) * D + d] = from_f32<T>(num / den);
        } else {
            const int64_t slot = (static_cast<int64_t>(row) * num_q_heads + hq) * num_parts + p;
            ws_o[slot * D + d] = num / den;
            if (d == 0) {
                ws_ml[2 * slot] = M;
                ws_ml[2 * slot + 1] = den;
            }
        }
    }
}

// Merges the partitions of sequences that needed more than one (grid: sequence x q head).
template <typename T, int D>
__global__ void __launch_bounds__(D) decode_simt_reduce_kernel(T* __restrict__ out,
                                                               const int32_t* __restrict__ seq_lens,
                                                               int32_t cap, int32_t num_q_heads,
                                                               int32_t part_tokens, int32_t num_parts,
                                                               const float* __restrict__ ws_o,
                                                               const float* __restrict__ ws_ml) {
    const int32_t s = blockIdx.x, hq = blockIdx.y, d = threadIdx.x;
    int32_t len = __ldg(seq_lens + s);
    len = len < 0 ? 0 : (len > cap ? cap : len);
    const int32_t parts = (len + part_tokens - 1) / part_tokens;
    if (parts <= 1) return;
    const int64_t slot0 = (static_cast<int64_t>(s) * num_q_heads + hq) * num_parts;
    float M = -INFINITY;
    for (int32_t p = 0; p < parts; ++p) M = fmaxf(M, ws_ml[2 * (slot0 + p)]);
    float num = 0.f, den = 0.f;
    for (int32_t p = 0; p < parts; ++p) {
        const float w = ws_ml[2 * (slot0 + p) + 1] * exp2f(ws_ml[2 * (slot0 + p)] - M);
        num = fmaf(w, ws_o[(slot0 + p) * D + d], num);
        den += w;
    }
    out[(static_cast<int64_t>(s) * num_q_heads + hq) * D + d] = from_f32<T>(num / den);
}

}  // namespace

template <typename T, int D>
static cudaError_t launch_simt_impl(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    const float scale_log2 = a.scale * kLog2e;
    float* ws_o = static_cast<float*>(a.workspace);
    float* ws_ml = ws_o + static_cast<size_t>(a.num_seqs) * a.num_q_heads * plan.num_partitions * D;
    dim3 grid(a.num_seqs, a.num_kv_heads * plan.head_chunks, plan.num_partitions);
    decode_simt_kernel<T, D><<<grid, kSimtThreads, 0, stream>>>(
        static_cast<T*>(a.out), static_cast<const T*>(a.q), static_cast<const T*>(a.k_cache),
        static_cast<const T*>(a.v_cache), a.block_table, a.max_blocks_per_seq, a.seq_lens, a.num_q_heads,
        a.num_kv_heads, a.num_blocks, scale_log2, plan.partition_tokens, plan.num_partitions, plan.head_chunks,
        ws_o, ws_ml, nullptr, a.num_seqs, block_size_log2(a.block_size) - 4, a.err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || plan.num_partitions == 1) return e;
    const int32_t cap = min(table_tokens(a.max_blocks_per_seq, block_size_log2(a.block_size) - 4),
                            plan.num_partitions * plan.partition_tokens);
    decode_simt_reduce_kernel<T, D><<<dim3(a.num_seqs, a.num_q_heads), D, 0, stream>>>(
        static_cast<T*>(a.out), a.seq_lens, cap, a.num_q_heads, plan.partition_tokens, plan.num_partitions, ws_o,
        ws_ml);
    return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t launch_simt_prefill(const PrefillArgs& a, int32_t total_rows, cudaStream_t stream) {
    // One CTA per (chunk row, kv head x head chunk), whole visible length: no workspace.
    const int32_t G = a.num_q_heads / a.num_kv_heads;
    const int32_t head_chunks = (G + kSimtHeads - 1) / kSimtHeads;
    const int32_t pt = max(kPageTokens, ((a.max_seq_len + kPageTokens - 1) / kPageTokens) * kPageTokens);
    dim3 grid(total_rows, a.num_kv_heads * head_chunks, 1);
    decode_simt_kernel<T, D><<<grid, kSimtThreads, 0, stream>>>(
        static_cast<T*>(a.out), static_cast<const T*>(a.q), static_cast<const T*>(a.k_cache),
        static_cast<const T*>(a.v_cache), a.block_table, a.max_blocks_per_seq, a.seq_lens, a.num_q_heads,
        a.num_kv_heads, a.num_blocks, a.scale * kLog2e, pt, 1, head_chunks, nullptr, nullptr, a.query_start_loc,
        a.num_seqs, block_size_log2(a.block_size) - 4, a.err);
    return cudaGetLastError();
}

cudaError_t launch_prefill_simt(const PrefillArgs& a, int32_t total_rows, cudaStream_t stream) {
    if (total_rows == 0 || a.num_seqs == 0) return cudaSuccess;
    if (a.dtype == PA_F32) {
        return a.head_dim == 128 ? launch_simt_prefill<float, 128>(a, total_rows, stream)
                                 : launch_simt_prefill<float, 64>(a, total_rows, stream);
    }
    return a.head_dim == 128 ? launch_simt_prefill<uint16_t, 128>(a, total_rows, stream)
                             : launch_simt_prefill<uint16_t, 64>(a, total_rows, stream);
}

cudaError_t launch_decode_simt(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    if (a.dtype == PA_F32) {
        return a.head_dim == 128 ? launch_simt_impl<float, 128>(a, plan, stream)
                                 : launch_simt_impl<float, 64>(a, plan, stream);
    }
    return a.head_dim == 128 ? launch_simt_impl<uint16_t, 128>(a, plan, stream)
                             : launch_simt_impl<uint16_t, 64>(a, plan, stream);
}

int simt_heads_per_cta() { return kSimtHeads; }

}  // namespace pa
