// Balanced persistent decode kernel for bf16 GQA groups of 4..16 q heads per kv head:
// TMA page staging, mma.sync, and a split-KV reduce done in place.
//
// Work list. The unit of work is one (sequence, kv head, logical block) page: 16 tokens x
// head_dim of K plus the same of V (8 KB at head_dim 128). Units are ordered sequence-major,
// then kv head, then page, so the units of one (sequence, kv head) "segment" are contiguous.
// Every CTA rebuilds the list's prefix sums from seq_lens with a block-wide scan and takes a
// contiguous slice of it (one persistent CTA per SM); inside the CTA each warp takes an equal
// contiguous sub-slice. The slices are equal to within one page whatever the mix of lengths,
// except that the last tenth of the CTAs, which start last when launches overlap, get a fixed
// number of pages fewer (Slices).
//
// Streaming. Each warp is an independent worker with its own ring of stages in shared memory.
// Lane 0 resolves a page's physical block through the block table ("My Understanding of vLLM
// and PagedAttention", "Block Table") and issues the page's K and V as one TMA tile copy each
// (128-byte swizzle; at head_dim 128 a 3-D box of 64 columns x 16 rows x 2 column halves, so the
// page lands as two 2 KB swizzled halves) completing on the stage's mbarrier; when the unit starts
// a new segment it also bulk-copies that segment's G query rows into the stage. Block ids are
// fetched 32 units ahead by the warp's lanes. The warp consumes a stage and refills it with
// the unit `stages` ahead. The math runs transposed on mma.sync m16n8k16 so that the page's 16
// keys fill the 16 rows: S^T = K Q^T (the G q heads that share the kv head as the 8 or 16
// columns, so each page is read once for the whole group), then O^T += V^T P^T with P^T
// brought into the B-operand layout by a register transpose (movmatrix); online softmax in
// registers, log2 domain. The unused tail of a sequence's last block may hold anything:
// its keys are masked to -inf and its V rows zeroed in shared memory before P V.
//
// Split-KV reduce, in three levels, all with the same log-sum-exp merge
//   M = max_p m_p,  w_p = l_p 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p :
//  1. a segment inside one warp's sub-slice is normalised and written from registers;
//  2. pieces cut by warp boundaries meet in shared memory after one CTA barrier; the groups
//     of pieces are listed (those also cut by the CTA range first) and shared out over the
//     CTA's warps;
//  3. segments cut by CTA boundaries leave one piece per CTA in the workspace; the warp that
//     counts the last piece (device-scope acquire-release counter per segment) merges them
//     and puts the counter back to zero.
//
// Variants: a block of 32, 64 or 128 tokens is walked as 2, 4 or 8 pages of 16 (sub_log2);
// APPEND fuses the step's new-token write (the page holding position len - 1 brings the new
// K/V rows, which the warp patches in and stores to the token's slot); a grid capped below
// the SM count (decode beside prefill) runs 10 warps per CTA; tables_ready moves the lengths
// scan and the first block-id loads before the grid-dependency wait.
#include <cuda.h>  // CUtensorMap (type only)
#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_trace.cuh"

namespace pa {
#ifdef PA_TRACE
static __device__ uint64_t g_trace[kTraceWords];
static __device__ uint32_t g_trace_counter;
#endif
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBalMaxGroup = 16;
constexpr int kBalMaxSeqs = 1024;  // per-sequence tables live in shared memory
constexpr uint32_t kLightBytes = 96u * 1024u;  // K/V bytes fewer for each of the last CTAs

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Stage: K page (D/64 swizzled 2 KB boxes), V page, then the segment's query rows; when the
// call appends each sequence's new token, then that token's K row, V row, its slot (int64) and
// the page's pool row (int32).
__host__ __device__ inline uint32_t bal_append_bytes(int D) { return 4u * D + 16u; }
__host__ __device__ inline uint32_t bal_stage_bytes(int D, int G, bool append) {
    return align_up(2u * kPageTokens * D * 2u + static_cast<uint32_t>(G) * D * 2u + (append ? bal_append_bytes(D) : 0u),
                    1024u);
}

struct BalLayout {
    uint32_t ring, piece0, piece_ml, meta, bars, flags, prefix, lens, total;
};

__host__ __device__ inline BalLayout bal_layout(int NW, int nst, uint32_t stage_bytes, int G, int D, int S) {
    BalLayout L;
    uint32_t o = 0;
    L.ring = o;      o += static_cast<uint32_t>(NW) * nst * stage_bytes;
    L.piece0 = o;    o += static_cast<uint32_t>(NW) * G * D * 4u;             // each warp's first piece
    L.piece_ml = o;  o += static_cast<uint32_t>(NW) * 2u * G * 2u * 4u;       // (m, l) of both pieces
    L.meta = o;      o += align_up(static_cast<uint32_t>(NW) * 2u * 4u * 2u + 16u, 16u);  // pieces, group list
    L.bars = o;      o += static_cast<uint32_t>(NW) * nst * 8u;
    L.flags = o;     o += 16u;
    L.prefix = o;    o += align_up((S + 1) * 4u, 16u);
    L.lens = o;      o += align_up(S * 4u, 16u);
    L.total = o + 1024u;  // base alignment slack
    return L;
}

struct BalWorkspace {
    int32_t* counter;  // [S * H_kv] finished CTA pieces per segment; zero between calls
    float* piece_o;    // [C][2][G][D] normalised partial outputs of CTA pieces
    float* piece_ml;   // [C][2][G][2] (max, sum) in the log2 domain
};

__host__ __device__ inline size_t bal_align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

__host__ __device__ inline size_t bal_ws_bytes(int S, int Hkv, int G, int D, int C) {
    return bal_align256(static_cast<size_t>(S) * Hkv * 4) + static_cast<size_t>(C) * 2 * G * D * 4 +
           static_cast<size_t>(C) * 2 * G * 2 * 4;
}

__host__ __device__ inline BalWorkspace bal_ws(void* base, int S, int Hkv, int G, int D, int C) {
    BalWorkspace w;
    char* p = static_cast<char*>(base);
    w.counter = reinterpret_cast<int32_t*>(p);
    p += bal_align256(static_cast<size_t>(S) * Hkv * 4);
    w.piece_o = reinterpret_cast<float*>(p);
    p += static_cast<size_t>(C) * 2 * G * D * 4;
    w.piece_ml = reinterpret_cast<float*>(p);
    return w;
}

// 2^x with the hardware approximation (relative error about 2^-22; 2^-inf = 0; results below
// 2^-126 flush to 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The work list's U units cut into C contiguous slices, one per CTA. With programmatic
// launches a grid's CTAs take the SMs in index order as the previous grid's CTAs leave them, so
// the highest-indexed CTAs start last, up to a few microseconds after the first ones. The last
// K CTAs (from cb = C - K on) therefore get d units fewer than the others: with A = U + K d,
// slice c starts at floor((c A - C max(0, c - cb) d) / C). Light slices are used only when each
// of them keeps at least one unit (U - cb d >= C); otherwise the slices are equal (K = d = 0).
struct Slices {
    int64_t U, A;
    int32_t C, cb, d;
    __host__ __device__ __forceinline__ void init(int64_t u, int32_t c, int32_t light, int32_t deficit) {
        U = u;
        C = c;
        cb = c - light;
        d = deficit;
        if (light <= 0 || light >= c || deficit <= 0 || u - static_cast<int64_t>(cb) * deficit < c) {
            cb = c;
            d = 0;
        }
        A = U + static_cast<int64_t>(C - cb) * d;
    }
    // first unit of slice c
    __host__ __device__ __forceinline__ int64_t start(int64_t c) const {
        const int64_t light = c > cb ? c - cb : 0;
        return (c * A - static_cast<int64_t>(C) * light * d) / C;
    }
    // the slice that holds unit u (the last one among slices that start at or before u)
    __host__ __device__ __forceinline__ int32_t owner(int64_t u) const {
        const int64_t c1 = ((u + 1) * C + A - 1) / A - 1;  // the answer if it is a full slice
        if (c1 < cb) return static_cast<int32_t>(c1);
        const int64_t den = U - static_cast<int64_t>(cb) * d;
        const int64_t c2 = ((u + 1 - static_cast<int64_t>(cb) * d) * C + den - 1) / den - 1;
        return static_cast<int32_t>(c2 < C - 1 ? c2 : C - 1);
    }
};

// Sequence s with prefix[s] <= u < prefix[s + 1].
__device__ __forceinline__ int32_t find_seq(const int32_t* prefix, int32_t S, int32_t u) {
    int32_t lo = 0, hi = S;
    while (hi - lo > 1) {
        const int32_t mid = (lo + hi) >> 1;
        if (prefix[mid] <= u) lo = mid; else hi = mid;
    }
    return lo;
}

// Position in the work list: sequence s, kv head h, page j of np pages, sequence length len.
struct Walker {
    int32_t s, h, j, np, len;
    __device__ __forceinline__ void at(const int32_t* prefix, const int32_t* lens, int32_t S, int32_t Hkv,
                                       int32_t u) {
        s = find_seq(prefix, S, u);
        np = (prefix[s + 1] - prefix[s]) / Hkv;
        const int32_t r = u - prefix[s];
        h = r / np;
        j = r - h * np;
        len = lens[s];
    }
    __device__ __forceinline__ void advance(const int32_t* prefix, const int32_t* lens, int32_t S, int32_t Hkv) {
        if (++j < np) return;
        j = 0;
        if (++h < Hkv) return;
        h = 0;
        do { ++s; } while (s < S && prefix[s + 1] == prefix[s]);
        if (s < S) {
            np = (prefix[s + 1] - prefix[s]) / Hkv;
            len = lens[s];
        }
    }
};

// 8-byte asynchronous copy global -> shared whose completion the mbarrier tracks: the arrive
// raises the barrier's pending count now and lowers it when the copy has landed.
__device__ __forceinline__ void async_copy8_tracked(void* smem_dst, const void* src, uint64_t* bar) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(smem_dst)), "l"(src) : "memory");
    asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void bulk_copy_g2s(void* smem_dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Bounded wait that does not give up early on the abort flag (used to drain in-flight copies).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > limit_ns) return;
    }
}

// Merge of a segment's CTA pieces by the warp that counted its last one. Pieces are those of
// the non-empty CTA slices w_first..w_last of W (slot 1 for w_first when the segment starts
// inside that slice). Heads go four at a time and pieces four at a time; lane l owns
// head_dim elements E*l..E*l+E-1. Every load of a batch (the pieces' (m, l) and their
// partial outputs) is issued before any is used, and a running maximum folds the batches:
//   M' = max(M, m_j),  den = den 2^(M - M') + sum_j l_j 2^(m_j - M'),  acc likewise with o_j.
template <int D>
__device__ __forceinline__ void merge_pieces(__nv_bfloat16* o, int32_t first_slot, int32_t w_first, int32_t w_last,
                                             int64_t U, int64_t W, int32_t G, const BalWorkspace& ws, int32_t lane,
                                             const PartOut& part, int64_t row0) {
    constexpr int E = D / 32;
    const bool may_be_empty = U < W;  // then the slices are equal
    for (int32_t g0 = 0; g0 < G; g0 += 4) {
        float M[4], den[4], acc[4][E];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            M[k] = -INFINITY;
            den[k] = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[k][e] = 0.f;
        }
        for (int32_t w0 = w_first; w0 <= w_last; w0 += 4) {
            float2 ml[4][4];
            float v[4][4][E];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int32_t w = w0 + j;
                bool ok = w <= w_last;
                if (ok && may_be_empty) ok = w * U / W < (w + 1) * U / W;
                const int64_t piece = static_cast<int64_t>(w) * 2 + (w == w_first ? first_slot : 0);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    if (ok && g0 + k < G) {
                        const int64_t pg = piece * G + g0 + k;
                        ml[j][k] = __ldcg(reinterpret_cast<const float2*>(ws.piece_ml + pg * 2));
                        const float* src = ws.piece_o + pg * D + lane * E;
                        if constexpr (E == 4) {
                            const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
                            v[j][k][0] = t.x; v[j][k][1] = t.y; v[j][k][2] = t.z; v[j][k][3] = t.w;
                        } else {
                            const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
                            v[j][k][0] = t.x; v[j][k][1] = t.y;
                        }
                    } else {
                        ml[j][k] = make_float2(-INFINITY, 0.f);
#pragma unroll
                        for (int e = 0; e < E; ++e) v[j][k][e] = 0.f;
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float Mn = M[k];
#pragma unroll
                for (int j = 0; j < 4; ++j) Mn = fmaxf(Mn, ml[j][k].x);
                const float sc = (M[k] == -INFINITY) ? 0.f : fast_exp2(M[k] - Mn);
                den[k] *= sc;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[k][e] *= sc;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float wj = (ml[j][k].x == -INFINITY) ? 0.f : ml[j][k].y * fast_exp2(ml[j][k].x - Mn);
                    den[k] += wj;
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[k][e] = fmaf(wj, v[j][k][e], acc[k][e]);
                }
                M[k] = Mn;
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (g0 + k < G) {
                const float inv = 1.f / den[k];
                if (part.o != nullptr) {  // a part: normalised fp32 row and its (max, sum)
                    float* po = part.o + (row0 + g0 + k) * D + lane * E;
#pragma unroll
                    for (int e = 0; e < E; ++e) po[e] = acc[k][e] * inv;
                    if (lane == 0) part.ml[row0 + g0 + k] = make_float2(M[k], den[k]);
                    continue;
                }
                uint32_t* dst = reinterpret_cast<uint32_t*>(o + (g0 + k) * D + lane * E);
                dst[0] = pack_bf16x2(acc[k][0] * inv, acc[k][1] * inv);
                if constexpr (E == 4) dst[1] = pack_bf16x2(acc[k][2] * inv, acc[k][3] * inv);
            }
        }
    }
}

// Adds one finished piece to a segment's counter; acquire-release at device scope, so the
// counting thread's warp saw its own piece stores (warp barrier before) and the last one to
// count sees every other piece (warp barrier after, in the caller).
__device__ __forceinline__ int32_t count_piece(int32_t* counter) {
    int32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
    return old;
}

// NH: groups of 8 q heads (G <= 8 * NH). APPEND: the call appends each sequence's new token
// (a separate instantiation, so plain decode carries none of its code).
template <int D, int NW, int NH, bool APPEND>
__global__ void __launch_bounds__(NW * 32, 1) decode_balanced_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ block_table,
    int32_t max_blocks, const int32_t* __restrict__ seq_lens, int32_t S, int32_t num_kv_heads, int32_t G,
    int32_t num_blocks, int32_t sub_log2, float scale_log2, int32_t nst, uint32_t stage_bytes, BalWorkspace ws,
    uint32_t* err, const int4* __restrict__ k_new, const int4* __restrict__ v_new,
    const int64_t* __restrict__ slot_mapping, int4* __restrict__ k_pool, int4* __restrict__ v_pool,
    int32_t tables_ready, int32_t pool_ready, uint64_t wait_limit_ns, int32_t drill, int32_t len_offset,
    PartOut part, int32_t light_ctas, int32_t light_units) {
    constexpr uint32_t kPage = kPageTokens * D * 2;
    constexpr uint32_t kHalves = D / 64;
    constexpr int KS = D / 16;  // k-steps over head_dim
    constexpr int E = D / 32;   // elements per lane in the merges
    constexpr int NTH = NW * 32;
    static_assert(NW <= 16, "level-2 reductions cover the pieces of at most 16 warps");
    constexpr int kPieceLanes = NW > 8 ? 16 : 8;  // lanes that can hold a group's pieces
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const BalLayout L = bal_layout(NW, nst, stage_bytes, G, D, S);
    float* piece0 = reinterpret_cast<float*>(smem + L.piece0);
    float* piece_ml = reinterpret_cast<float*>(smem + L.piece_ml);
    int32_t* meta = reinterpret_cast<int32_t*>(smem + L.meta);  // [NW][2] segment of each piece
    int32_t* glist = meta + 2 * NW;                                  // [2 NW] groups to merge (owner slot)
    int32_t* gcount = glist + 2 * NW;                                // [2] crossing / internal group counts
    uint64_t* bars_all = reinterpret_cast<uint64_t*>(smem + L.bars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.flags);
    int32_t* prefix = reinterpret_cast<int32_t*>(smem + L.prefix);
    int32_t* lens = reinterpret_cast<int32_t*>(smem + L.lens);

    const int32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // keys [len_offset, len) of each sequence; the caller's table row begins at its
    // len_offset / block_size-th entry
    const int32_t cap = table_tokens(max_blocks, sub_log2) - len_offset;
    const int32_t Hq = G * num_kv_heads;
    PA_TRACE_DECL
    PA_TRACE_BEGIN(g_trace_counter);
    PA_TRACE_STAMP(g_trace, 0);

    // Inputs may come from the kernel before this one in the stream (programmatic launch). When
    // the caller says that kernel writes neither seq_lens nor the block table (tables_ready),
    // the lengths scan and the first block-id loads run before the wait, overlapping its tail;
    // everything else (pool, queries, new rows, output, workspace) is touched after it.
    // Right after its wait each thread also lets the next kernel's grid be launched: its CTAs
    // take an SM as soon as one of ours leaves it (a second decode CTA does not fit beside this
    // one) and wait there for this grid to complete, so the launch latency hides behind our
    // merge tail. Triggering only after the wait means that every kernel before this one has
    // completed when the next one starts.
    auto dep_wait = [&]() {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    };
    // The tensor maps are kernel parameters, which no earlier kernel writes: fetch them now.
    if (tid == 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    if (!tables_ready) dep_wait();

    // ---- prologue: clamped lengths and units per sequence, block-wide exclusive scan -------
    {
        const int32_t per = (S + NTH - 1) / NTH;
        const int32_t b = min(S, tid * per), e = min(S, b + per);
        int32_t local = 0;
        for (int32_t s = b; s < e; ++s) {
            int32_t len = __ldg(seq_lens + s) - len_offset;
            if (len < 0 || len > cap) {
                if (blockIdx.x == 0) raise_error(err, PA_DEVERR_LEN_RANGE);
                len = len < 0 ? 0 : cap;
            }
            lens[s] = len;
            local += ((len + kPageTokens - 1) / kPageTokens) * num_kv_heads;
        }
        int32_t incl = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        __shared__ int32_t warp_tot[NW];
        if (lane == 31) warp_tot[warp] = incl;
        if (lane == 0) {
            meta[warp * 2] = -1;
            meta[warp * 2 + 1] = -1;
            if (warp == 0) gcount[0] = gcount[1] = 0;
            for (int i = 0; i < nst; ++i) mbar_init(&bars_all[warp * nst + i], 1);
        }
        if (tid == 0) *abort_flag = 0;
        fence_mbarrier_init();
        __syncthreads();
        int32_t base = 0;
        for (int w = 0; w < warp; ++w) base += warp_tot[w];
        int32_t run = base + incl - local;
        for (int32_t s = b; s < e; ++s) {
            prefix[s] = run;
            run += ((lens[s] + kPageTokens - 1) / kPageTokens) * num_kv_heads;
        }
        if (tid == NTH - 1) prefix[S] = base + incl;
        __syncthreads();
    }
    PA_TRACE_STAMP(g_trace, 1);
    if (len_offset > 0) {
        // every table row must begin with row 0's prefix blocks (the caller's rows start
        // len_offset / block_size entries before the ones this kernel walks)
        const int32_t pb = len_offset >> (sub_log2 + 4);
        const int32_t* bt0 = block_table - pb;
        const int64_t n_ids = static_cast<int64_t>(S) * pb;
        for (int64_t i = static_cast<int64_t>(blockIdx.x) * NTH + tid; i < n_ids; i += static_cast<int64_t>(gridDim.x) * NTH) {
            const int64_t s = i / pb, j = i - s * pb;
            if (__ldg(bt0 + s * max_blocks + j) != __ldg(bt0 + j)) raise_error(err, PA_DEVERR_PREFIX_MISMATCH);
        }
    }

    const int64_t U = prefix[S];
    const int64_t C = gridDim.x;
    // Append (k_new != nullptr): sequence i's token at position len_i - 1 is new. The warp that
    // attends over the page holding that position receives the token's K/V rows with the page,
    // uses them for that row and writes them to slot_mapping[i]: no kernel waits on its own pool
    // writes, and the writes cost no load latency on the streaming path.
    constexpr bool append = APPEND;
    constexpr int32_t CPR = D * 2 / 16;  // 16-byte chunks per K or V row
    const int32_t bs_log2 = sub_log2 + 4;
    // sequences without keys get zero rows (spread over the CTAs); with append their new rows
    // are written here
    for (int32_t s = blockIdx.x; s < S; s += gridDim.x) {
        if (lens[s] != 0) continue;
        if (tables_ready) dep_wait();
        if (part.o != nullptr) {  // an empty part: zero output, weight zero
            for (int32_t i = tid; i < Hq * D; i += NTH) part.o[static_cast<int64_t>(s) * Hq * D + i] = 0.f;
            for (int32_t i = tid; i < Hq; i += NTH) part.ml[static_cast<int64_t>(s) * Hq + i] = make_float2(-INFINITY, 0.f);
        } else {
            uint32_t* z = reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(s) * Hq * D);
            for (int32_t i = tid; i < Hq * D / 2; i += NTH) z[i] = 0u;
        }
        if (append) {
            const int64_t slot = __ldg(slot_mapping + s);
            if (slot >= (static_cast<int64_t>(num_blocks) << bs_log2)) {
                if (tid == 0) raise_error(err, PA_DEVERR_SLOT_RANGE);
            } else if (slot >= 0) {
                const int64_t blk = slot >> bs_log2, off = slot - (blk << bs_log2);
                for (int32_t i = tid; i < num_kv_heads * CPR; i += NTH) {
                    const int32_t h = i / CPR, c = i - h * CPR;
                    const int64_t dst = (((blk * num_kv_heads + h) << bs_log2) + off) * CPR + c;
                    const int64_t src = (static_cast<int64_t>(s) * num_kv_heads + h) * CPR + c;
                    k_pool[dst] = __ldg(k_new + src);
                    v_pool[dst] = __ldg(v_new + src);
                }
            }
        }
    }
    int32_t u0, u1;
    {
        Slices sl;
        sl.init(U, static_cast<int32_t>(C), light_ctas, light_units);
        u0 = static_cast<int32_t>(sl.start(blockIdx.x));
        u1 = static_cast<int32_t>(sl.start(blockIdx.x + 1));
    }
    if (u0 >= u1) return;  // uniform over the CTA
    const int32_t n_cta = u1 - u0;
    const int32_t a_w = u0 + static_cast<int32_t>((static_cast<int64_t>(warp) * n_cta) / NW);
    const int32_t b_w = u0 + static_cast<int32_t>((static_cast<int64_t>(warp + 1) * n_cta) / NW);
    const int32_t n = b_w - a_w;
    uint8_t* ring = smem + L.ring + static_cast<uint32_t>(warp) * nst * stage_bytes;
    const uint32_t ring_u32 = smem_u32(ring);
    uint64_t* bars = bars_all + warp * nst;
    const int32_t gid = lane >> 2, tig = lane & 3;

    int32_t consumed = 0, issued = 0;
    if (n > 0) {
        // Block-table row of unit a_w + 32 k + lane (pool row of its (block, kv head) page).
        auto lane_row = [&](int32_t k) -> int32_t {
            const int32_t u = a_w + 32 * k + lane;
            if (u >= b_w) return 0;
            const int32_t s = find_seq(prefix, S, u);
            const int32_t np = (prefix[s + 1] - prefix[s]) / num_kv_heads;
            const int32_t r = u - prefix[s];
            const int32_t h = r / np, j = r - h * np;
            int32_t phys = __ldg(block_table + static_cast<int64_t>(s) * max_blocks + (j >> sub_log2));
            if (phys < 0 || phys >= num_blocks) {
                raise_error(err, PA_DEVERR_BLOCK_RANGE);
                phys = 0;
            }
            return ((((phys * num_kv_heads + h) << sub_log2) + (j & ((1 << sub_log2) - 1))) * kPageTokens);
        };
        int32_t kc = 0;
        int32_t id_cur = lane_row(0);
        int32_t id_nxt = n > 32 ? lane_row(1) : 0;
        Walker wi;
        wi.at(prefix, lens, S, num_kv_heads, a_w);
        // KV pages are read once per call: let them leave L2 first, ahead of the block table,
        // queries, lengths and this kernel's own code.
        const uint64_t kv_policy = l2_policy_evict_first();
        const uint32_t qbytes = static_cast<uint32_t>(G) * D * 2u;

        // Pool row of unit t's page (block ids fetched 32 units ahead); warp-uniform.
        auto page_row = [&](int32_t t) -> int32_t {
            if ((t >> 5) == kc + 1) {
                ++kc;
                id_cur = id_nxt;
                id_nxt = 32 * (kc + 1) < n ? lane_row(kc + 1) : 0;
            }
            return __shfl_sync(0xffffffffu, id_cur, t & 31);
        };
        // Bytes that arrive in a stage besides the K and V pages: the segment's query rows with
        // its first page, the new token's rows with the page that holds position len - 1.
        // With the wait drill on, the warp holding unit 0 announces 16 bytes more for its first
        // stage than any copy brings: that stage never completes and its wait runs out.
        const uint32_t drill_bytes = (drill && a_w == 0) ? 16u : 0u;
        auto extra_bytes = [&](int32_t t, const Walker& w) -> uint32_t {
            const bool seg_first = (t == 0) || (w.j == 0);
            const bool new_row = append && w.j == w.np - 1;
            return (seg_first ? qbytes : 0u) + (new_row ? 4u * D : 0u) + (t == 0 ? drill_bytes : 0u);
        };
        // The page copies of unit t (lane 0). With `arrive` the stage's single arrival is made
        // here together with every byte it expects; without it only the pages' bytes are
        // announced, and issue_rest() arrives later.
        auto issue_pages = [&](int32_t t, int32_t row, const Walker& w, bool arrive) {
            const int32_t st = t % nst;
            uint8_t* stage = ring + static_cast<uint32_t>(st) * stage_bytes;
            if (append && w.j == w.np - 1)  // the page's pool row, behind the query rows and new K/V
                *reinterpret_cast<int32_t*>(stage + 2u * kPage + qbytes + 4u * D + 8u) = row;
            if (arrive) mbar_arrive_expect_tx(&bars[st], 2u * kPage + extra_bytes(t, w));
            else mbar_expect_tx(&bars[st], 2u * kPage);
            if constexpr (kHalves == 2) {  // both 64-column halves in one box
                tma_load_3d_hint(stage, &tm_k, 0, row, 0, &bars[st], kv_policy);
                tma_load_3d_hint(stage + kPage, &tm_v, 0, row, 0, &bars[st], kv_policy);
            } else {
                tma_load_2d_hint(stage, &tm_k, 0, row, &bars[st], kv_policy);
                tma_load_2d_hint(stage + kPage, &tm_v, 0, row, &bars[st], kv_policy);
            }
        };
        // The rest of unit t's stage (lane 0): the segment's query rows, the new token's K/V rows
        // and its slot; `arrive` makes the stage's arrival (pages already announced).
        auto issue_rest = [&](int32_t t, const Walker& w, bool arrive) {
            const int32_t st = t % nst;
            uint8_t* stage = ring + static_cast<uint32_t>(st) * stage_bytes;
            if (arrive) mbar_arrive_expect_tx(&bars[st], extra_bytes(t, w));
            if (append && w.j == w.np - 1) {
                uint8_t* ex = stage + 2u * kPage + qbytes;
                async_copy8_tracked(ex + 4u * D, slot_mapping + w.s, &bars[st]);
                const int64_t r = static_cast<int64_t>(w.s) * num_kv_heads + w.h;
                bulk_copy_g2s(ex, k_new + r * CPR, D * 2u, &bars[st]);
                bulk_copy_g2s(ex + D * 2u, v_new + r * CPR, D * 2u, &bars[st]);
            }
            if ((t == 0) || (w.j == 0))
                bulk_copy_g2s(stage + 2u * kPage, q + (static_cast<int64_t>(w.s) * Hq + w.h * G) * D, qbytes, &bars[st]);
        };
        auto issue = [&](int32_t t) {  // warp-uniform
            const int32_t row = page_row(t);
            if (lane == 0 && !*abort_flag) {
                issue_pages(t, row, wi, true);
                issue_rest(t, wi, false);
            }
            if (t < 8) PA_TRACE_STAMP(g_trace, 24 + t);
            wi.advance(prefix, lens, S, num_kv_heads);
            issued = t + 1;
        };

        const int32_t pre = min(nst, n);
        if (pool_ready) {
            // The pool pages do not come from the kernel before this one: start the first
            // stages' page copies now and only the rest of each stage after the wait. Each
            // stage's phase completes only after its arrival (made after the wait), whatever
            // the order in which the bytes land.
            for (int32_t t = 0; t < pre; ++t) {
                const int32_t row = page_row(t);
                if (lane == 0) issue_pages(t, row, wi, false);
                if (t < 8) PA_TRACE_STAMP(g_trace, 24 + t);
                wi.advance(prefix, lens, S, num_kv_heads);
            }
            dep_wait();  // from here on: queries, new rows, output, workspace
            PA_TRACE_STAMP(g_trace, 2);
            Walker wq;
            wq.at(prefix, lens, S, num_kv_heads, a_w);
            for (int32_t t = 0; t < pre; ++t) {
                if (lane == 0) issue_rest(t, wq, true);
                wq.advance(prefix, lens, S, num_kv_heads);
            }
            issued = pre;
        } else {
            if (tables_ready) dep_wait();  // from here on: pool, queries, new rows, output
            PA_TRACE_STAMP(g_trace, 2);
            for (int32_t t = 0; t < pre; ++t) issue(t);
        }
        PA_TRACE_STAMP(g_trace, 3);

        Walker wc;
        wc.at(prefix, lens, S, num_kv_heads, a_w);
        constexpr int NMT = D / 16;  // m-tiles of O^T (16 head_dim rows each)
        // Fragment ownership (gid = lane / 4, tig = lane % 4):
        //   qb[nh][ks]   Q^T as B: head 8 nh + gid, dims 16 ks + 2 tig (+1) and + 8
        //   sc[nh][e]    S^T: key gid + 8 (e / 2), head 8 nh + 2 tig + e % 2
        //   acc[nh][mt]  O^T: head_dim 16 mt + gid + 8 (e / 2), head 8 nh + 2 tig + e % 2
        //   mh, lh       running max and partial sum of heads 8 nh + 2 tig + {0, 1}
        uint32_t qb[NH][KS][2];
        float acc[NH][NMT][4];
        float mh[NH][2], lh[NH][2];
        int32_t t_first = 0;

        for (int32_t t = 0; t < n; ++t) {
            const int32_t st = t % nst;
            const bool landed =
                mbar_wait_bounded(&bars[st], static_cast<uint32_t>(t / nst) & 1u, abort_flag, wait_limit_ns);
            if (!__all_sync(0xffffffffu, landed)) {  // lanes agree before any warp-wide step
                if (lane == 0) {
                    if (!*abort_flag) raise_error(err, PA_DEVERR_WAIT_TIMEOUT);
                    *abort_flag = 1;
                }
                __syncwarp();
                break;
            }
            consumed = t + 1;
            if (t == 0) PA_TRACE_STAMP(g_trace, 4);
            if (t < 8) PA_TRACE_STAMP(g_trace, 16 + t);
            uint8_t* stage = ring + static_cast<uint32_t>(st) * stage_bytes;
            const uint32_t k_u32 = ring_u32 + static_cast<uint32_t>(st) * stage_bytes;
            const uint32_t v_u32 = k_u32 + kPage;
            const bool seg_first = (t == 0) || (wc.j == 0);
            if (seg_first) {
                // the segment's G query rows were copied into this stage with the page
                const __nv_bfloat16* qs = reinterpret_cast<const __nv_bfloat16*>(stage + 2u * kPage);
#pragma unroll
                for (int nh = 0; nh < NH; ++nh) {
                    const int32_t head = nh * 8 + gid;
                    const bool valid = head < G;
#pragma unroll
                    for (int ks = 0; ks < KS; ++ks) {
                        const int c0 = ks * 16 + tig * 2;
                        qb[nh][ks][0] = valid ? *reinterpret_cast<const uint32_t*>(qs + head * D + c0) : 0u;
                        qb[nh][ks][1] = valid ? *reinterpret_cast<const uint32_t*>(qs + head * D + c0 + 8) : 0u;
                    }
#pragma unroll
                    for (int mt = 0; mt < NMT; ++mt) acc[nh][mt][0] = acc[nh][mt][1] = acc[nh][mt][2] = acc[nh][mt][3] = 0.f;
                    mh[nh][0] = mh[nh][1] = -INFINITY;
                    lh[nh][0] = lh[nh][1] = 0.f;
                }
                t_first = t;
            }
            const int32_t ntok = min(kPageTokens, wc.len - wc.j * kPageTokens);
            if (ntok < kPageTokens) {
                // zero the V rows of the unused tail so that p = 0 contributes exactly nothing
                const int32_t rows = kPageTokens - ntok;
                for (int32_t c = lane; c < rows * 8 * static_cast<int32_t>(kHalves); c += 32) {
                    const int32_t hf = c / (rows * 8), rem = c - hf * rows * 8;
                    *reinterpret_cast<int4*>(stage + kPage + hf * 2048u + (ntok + rem / 8) * 128u + (rem % 8) * 16u) =
                        make_int4(0, 0, 0, 0);
                }
                __syncwarp();
            }
            const bool new_row = append && wc.j == wc.np - 1;
            if (new_row) {
                // row ntok - 1 is the new token: take its K/V from the appended rows and write
                // them to the token's slot
                const uint8_t* ex = stage + 2u * kPage + static_cast<uint32_t>(G) * D * 2u;
                const int64_t slot = *reinterpret_cast<const int64_t*>(ex + 4u * D);
                const int64_t want = *reinterpret_cast<const int32_t*>(ex + 4u * D + 8u) + (ntok - 1);
                int64_t dst_row = -1;
                if (slot >= 0 && slot < (static_cast<int64_t>(num_blocks) << bs_log2)) {
                    const int64_t blk = slot >> bs_log2;
                    dst_row = ((blk * num_kv_heads + wc.h) << bs_log2) + (slot - (blk << bs_log2));
                } else if (slot >= 0 && lane == 0) {
                    raise_error(err, PA_DEVERR_SLOT_RANGE);
                }
                if (dst_row != want && lane == 0) raise_error(err, PA_DEVERR_APPEND_SLOT);
                if (lane < 2 * CPR) {
                    const int32_t kv = lane / CPR, c = lane - kv * CPR;
                    const int4 val = *reinterpret_cast<const int4*>(ex + kv * D * 2u + c * 16u);
                    *reinterpret_cast<int4*>(stage + kv * kPage + (c >> 3) * 2048u +
                                             sw128_offset(static_cast<uint32_t>(ntok - 1), c & 7u)) = val;
                    if (dst_row >= 0) (kv ? v_pool : k_pool)[dst_row * CPR + c] = val;
                }
                __syncwarp();
            }

            // S^T = K Q^T: rows = the page's 16 keys, columns = q heads
            const uint32_t mat = lane >> 3, r8 = lane & 7;
            float sc[NH][4];
#pragma unroll
            for (int nh = 0; nh < NH; ++nh) sc[nh][0] = sc[nh][1] = sc[nh][2] = sc[nh][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                // A fragments: matrix mat = (keys 8 (mat % 2) .., 16-byte chunk 2 ks + mat / 2)
                const uint32_t key = r8 + 8u * (mat & 1u), chunk = ks * 2 + (mat >> 1);
                uint32_t a[4];
                ldsm_x4(k_u32 + (chunk >> 3) * 2048u + sw128_offset(key, chunk & 7u), a[0], a[1], a[2], a[3]);
#pragma unroll
                for (int nh = 0; nh < NH; ++nh) mma_16816(sc[nh], a, qb[nh][ks][0], qb[nh][ks][1]);
            }
            // online softmax per head (column) in the log2 domain: reduce over the 16 keys =
            // the two rows a thread holds and the 8 lanes with the same tig
            float mx[NH][2];
#pragma unroll
            for (int nh = 0; nh < NH; ++nh) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int32_t k_in = gid + 8 * (e >> 1);
                    sc[nh][e] = k_in < ntok ? sc[nh][e] * scale_log2 : -INFINITY;
                }
                mx[nh][0] = fmaxf(sc[nh][0], sc[nh][2]);
                mx[nh][1] = fmaxf(sc[nh][1], sc[nh][3]);
            }
#pragma unroll
            for (int off = 4; off < 32; off <<= 1)
#pragma unroll
                for (int nh = 0; nh < NH; ++nh) {
                    mx[nh][0] = fmaxf(mx[nh][0], __shfl_xor_sync(0xffffffffu, mx[nh][0], off));
                    mx[nh][1] = fmaxf(mx[nh][1], __shfl_xor_sync(0xffffffffu, mx[nh][1], off));
                }
            uint32_t pb[NH][2];
#pragma unroll
            for (int nh = 0; nh < NH; ++nh) {
                float cc[2];
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const float mn = fmaxf(mh[nh][hh], mx[nh][hh]);
                    cc[hh] = fast_exp2(mh[nh][hh] - mn);
                    mh[nh][hh] = mn;
                }
                float p[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) p[e] = fast_exp2(sc[nh][e] - mh[nh][e & 1]);
                lh[nh][0] = lh[nh][0] * cc[0] + p[0] + p[2];
                lh[nh][1] = lh[nh][1] * cc[1] + p[1] + p[3];
#pragma unroll
                for (int mt = 0; mt < NMT; ++mt) {
                    acc[nh][mt][0] *= cc[0];
                    acc[nh][mt][1] *= cc[1];
                    acc[nh][mt][2] *= cc[0];
                    acc[nh][mt][3] *= cc[1];
                }
                // P^T as the B operand of O^T += V^T P^T: transpose the two 8 x 8 (key, head)
                // blocks held in the accumulator layout
                pb[nh][0] = movmatrix_trans(pack_bf16x2(p[0], p[1]));
                pb[nh][1] = movmatrix_trans(pack_bf16x2(p[2], p[3]));
            }
            // O^T += V^T P^T: rows = head_dim (16 per m-tile), columns = q heads, k = keys
#pragma unroll
            for (int mt = 0; mt < NMT; ++mt) {
                // A fragments (transposed loads): matrix mat = (keys 8 (mat / 2) .., chunk 2 mt + mat % 2)
                const uint32_t key = r8 + 8u * (mat >> 1), chunk = mt * 2 + (mat & 1u);
                uint32_t a[4];
                ldsm_x4_trans(v_u32 + (chunk >> 3) * 2048u + sw128_offset(key, chunk & 7u), a[0], a[1], a[2], a[3]);
#pragma unroll
                for (int nh = 0; nh < NH; ++nh) mma_16816(acc[nh][mt], a, pb[nh][0], pb[nh][1]);
            }

            const bool seg_last = (t == n - 1) || (wc.j == wc.np - 1);
            if (seg_last) {
                float Lh[NH][2];
#pragma unroll
                for (int nh = 0; nh < NH; ++nh) {
                    Lh[nh][0] = lh[nh][0];
                    Lh[nh][1] = lh[nh][1];
                }
#pragma unroll
                for (int off = 4; off < 32; off <<= 1)
#pragma unroll
                    for (int nh = 0; nh < NH; ++nh) {
                        Lh[nh][0] += __shfl_xor_sync(0xffffffffu, Lh[nh][0], off);
                        Lh[nh][1] += __shfl_xor_sync(0xffffffffu, Lh[nh][1], off);
                    }
                const int32_t seg_a = prefix[wc.s] + wc.h * wc.np, seg_b = seg_a + wc.np;
                if (seg_a >= a_w && seg_b <= b_w) {
                    // whole segment inside this warp: normalise and write out
                    const int64_t row0 = static_cast<int64_t>(wc.s) * Hq + wc.h * G;
                    __nv_bfloat16* o = out + row0 * D;
#pragma unroll
                    for (int nh = 0; nh < NH; ++nh)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int32_t head = nh * 8 + tig * 2 + hh;
                            if (head >= G) continue;
                            const float inv = 1.f / Lh[nh][hh];
                            if (part.o != nullptr) {  // a part: normalised fp32 row, (max, sum)
                                float* prow = part.o + (row0 + head) * D + gid;
#pragma unroll
                                for (int mt = 0; mt < NMT; ++mt) {
                                    prow[mt * 16] = acc[nh][mt][hh] * inv;
                                    prow[mt * 16 + 8] = acc[nh][mt][2 + hh] * inv;
                                }
                                if (gid == 0) part.ml[row0 + head] = make_float2(mh[nh][hh], Lh[nh][hh]);
                                continue;
                            }
                            __nv_bfloat16* orow = o + head * D + gid;
#pragma unroll
                            for (int mt = 0; mt < NMT; ++mt) {
                                orow[mt * 16] = __float2bfloat16_rn(acc[nh][mt][hh] * inv);
                                orow[mt * 16 + 8] = __float2bfloat16_rn(acc[nh][mt][2 + hh] * inv);
                            }
                        }
                } else {
                    // piece of a segment cut by the warp's sub-slice, kept for the CTA merge:
                    // slot 0 = the sub-slice's first segment (own buffer), slot 1 = its last
                    // one, finalised with the last unit, when the warp's ring is idle
                    const int slot = (t_first == 0) ? 0 : 1;
                    __syncwarp();
                    float* pa_acc = slot == 0 ? piece0 + static_cast<uint32_t>(warp) * G * D
                                              : reinterpret_cast<float*>(ring);
#pragma unroll
                    for (int nh = 0; nh < NH; ++nh)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const int32_t head = nh * 8 + tig * 2 + hh;
                            if (head >= G) continue;
                            float* prow = pa_acc + head * D + gid;
#pragma unroll
                            for (int mt = 0; mt < NMT; ++mt) {
                                prow[mt * 16] = acc[nh][mt][hh];
                                prow[mt * 16 + 8] = acc[nh][mt][2 + hh];
                            }
                            if (gid == 0)
                                *reinterpret_cast<float2*>(piece_ml + ((warp * 2 + slot) * G + head) * 2) =
                                    make_float2(mh[nh][hh], Lh[nh][hh]);
                        }
                    if (lane == 0) meta[warp * 2 + slot] = wc.s * num_kv_heads + wc.h;
                }
            }
            __syncwarp();
            if (ntok < kPageTokens || new_row) fence_proxy_async_shared();  // generic writes before the next copy
            if (t + nst < n) issue(t + nst);
            wc.advance(prefix, lens, S, num_kv_heads);
        }
        PA_TRACE_STAMP(g_trace, 5);
        PA_TRACE_AT(g_trace, 12, static_cast<uint64_t>(n));
        // after an abort: let the copies already issued land before the CTA can exit
        if (consumed < issued && lane == 0) {
            for (int32_t u = consumed; u < issued; ++u)
                mbar_drain(&bars[u % nst], static_cast<uint32_t>(u / nst) & 1u, wait_limit_ns);
        }
    }
    if (tables_ready && n <= 0) dep_wait();  // warps without pages still merge and write
    __syncthreads();
    PA_TRACE_STAMP(g_trace, 6);
    if (*abort_flag) return;

    // ---- level 2: merge the pieces of segments cut between this CTA's warps ----------------
    // A group is the run of pieces of one segment over consecutive warps of the CTA, named by
    // the slot of its last piece; lane i of the warp that merges it holds the group's i-th
    // piece counted from the end.
    auto warp_len = [&](int32_t w2) {
        return static_cast<int32_t>((static_cast<int64_t>(w2 + 1) * n_cta) / NW -
                                    (static_cast<int64_t>(w2) * n_cta) / NW);
    };
    // List the groups by their owner slot: those cut by the CTA range too (they go on to the
    // workspace merge, level 3) first, from the front, the others from the back; then the warps
    // share them out, so two expensive groups rarely land on one warp.
    if (lane == 0) {
        for (int32_t s0 = 0; s0 < 2; ++s0) {
            const int32_t seg = meta[warp * 2 + s0];
            if (seg < 0) continue;
            int32_t nxt = warp + 1;  // next warp of the CTA with units
            while (nxt < NW && warp_len(nxt) == 0) ++nxt;
            if (nxt < NW && meta[nxt * 2] == seg) continue;  // the group goes on in a later warp
            const int32_t sq = seg / num_kv_heads, hq = seg - sq * num_kv_heads;
            const int32_t npq = (prefix[sq + 1] - prefix[sq]) / num_kv_heads;
            const int32_t sa = prefix[sq] + hq * npq;
            const bool crossing = sa < u0 || sa + npq > u1;
            if (crossing) glist[atomicAdd(&gcount[0], 1)] = warp * 2 + s0;
            else glist[2 * NW - 1 - atomicAdd(&gcount[1], 1)] = warp * 2 + s0;
        }
    }
    __syncthreads();
    PA_TRACE_STAMP(g_trace, 7);
    const int32_t n_cross = gcount[0], n_groups = gcount[0] + gcount[1];
#ifdef PA_TRACE
    uint64_t tr_groups = 0, tr_l3 = 0;
#endif
    for (int32_t gi = warp; gi < n_groups; gi += NW) {
        const int32_t owner = glist[gi < n_cross ? gi : 2 * NW - 1 - (gi - n_cross)];
        const int32_t ow = owner >> 1, s0 = owner & 1;
        const int32_t seg = meta[owner];
        int32_t my_slot = lane == 0 ? owner : -1;
        int32_t nm = 1;
        if (s0 == 0) {  // the segment may have begun in earlier warps
            for (int32_t w2 = ow - 1; w2 >= 0; --w2) {
                if (warp_len(w2) == 0) continue;
                const int32_t slot2 = meta[w2 * 2 + 1] == seg ? w2 * 2 + 1 : (meta[w2 * 2] == seg ? w2 * 2 : -1);
                if (slot2 < 0) break;
                if (lane == nm) my_slot = slot2;
                ++nm;
                if (slot2 & 1) break;  // the segment begins inside warp w2
            }
        }
        const int32_t s = seg / num_kv_heads, h = seg - s * num_kv_heads;
        const int32_t np = (prefix[s + 1] - prefix[s]) / num_kv_heads;
        const int32_t seg_a = prefix[s] + h * np, seg_b = seg_a + np;
        const bool complete = seg_a >= u0 && seg_b <= u1;
        const int64_t cpiece = static_cast<int64_t>(blockIdx.x) * 2 + (seg_a <= u0 ? 0 : 1);
        // four heads at a time, their shuffle chains interleaved; pieces hold unnormalised
        // sums, so piece i weighs 2^(m_i - M) / sum_i l_i 2^(m_i - M)
        for (int32_t g0 = 0; g0 < G; g0 += 4) {
            float mk[4], lk[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                mk[k] = -INFINITY;
                lk[k] = 0.f;
                if (my_slot >= 0 && g0 + k < G) {
                    const float2 ml = *reinterpret_cast<const float2*>(piece_ml + (my_slot * G + g0 + k) * 2);
                    mk[k] = ml.x;
                    lk[k] = ml.y;
                }
            }
            float Mk[4], dk[4], wk[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) Mk[k] = mk[k];
#pragma unroll
            for (int off = kPieceLanes / 2; off > 0; off >>= 1)  // a group has at most NW pieces
#pragma unroll
                for (int k = 0; k < 4; ++k) Mk[k] = fmaxf(Mk[k], __shfl_xor_sync(0xffffffffu, Mk[k], off));
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                wk[k] = my_slot >= 0 ? fast_exp2(mk[k] - Mk[k]) : 0.f;
                dk[k] = lk[k] * wk[k];
            }
#pragma unroll
            for (int off = kPieceLanes / 2; off > 0; off >>= 1)
#pragma unroll
                for (int k = 0; k < 4; ++k) dk[k] += __shfl_xor_sync(0xffffffffu, dk[k], off);
#pragma unroll
            for (int k = 0; k < 4; ++k) wk[k] = __fdividef(wk[k], dk[k]);
            float v[4][E];
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int e = 0; e < E; ++e) v[k][e] = 0.f;
            for (int32_t i = 0; i < nm; ++i) {
                const int32_t si = __shfl_sync(0xffffffffu, my_slot, i);
                const float* a = ((si & 1) ? reinterpret_cast<const float*>(smem + L.ring + static_cast<uint32_t>(si >> 1) *
                                                                                              nst * stage_bytes)
                                           : piece0 + static_cast<uint32_t>(si >> 1) * G * D) +
                                 lane * E;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float wi = __shfl_sync(0xffffffffu, wk[k], i);
                    if (g0 + k < G) {
                        const float* ak = a + (g0 + k) * D;
                        if constexpr (E == 4) {
                            const float4 t = *reinterpret_cast<const float4*>(ak);
                            v[k][0] = fmaf(wi, t.x, v[k][0]); v[k][1] = fmaf(wi, t.y, v[k][1]);
                            v[k][2] = fmaf(wi, t.z, v[k][2]); v[k][3] = fmaf(wi, t.w, v[k][3]);
                        } else {
                            const float2 t = *reinterpret_cast<const float2*>(ak);
                            v[k][0] = fmaf(wi, t.x, v[k][0]); v[k][1] = fmaf(wi, t.y, v[k][1]);
                        }
                    }
                }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int32_t g = g0 + k;
                if (g >= G) continue;
                if (complete && part.o != nullptr) {
                    // a part: normalised fp32 row and (max, sum) (lane 0 holds them: it is one of
                    // the lanes the reductions above reach)
                    const int64_t row = static_cast<int64_t>(s) * Hq + h * G + g;
                    float* dst = part.o + row * D + lane * E;
#pragma unroll
                    for (int e = 0; e < E; ++e) dst[e] = v[k][e];
                    if (lane == 0) part.ml[row] = make_float2(Mk[k], dk[k]);
                } else if (complete) {
                    uint32_t* dst =
                        reinterpret_cast<uint32_t*>(out + (static_cast<int64_t>(s) * Hq + h * G + g) * D + lane * E);
                    dst[0] = pack_bf16x2(v[k][0], v[k][1]);
                    if constexpr (E == 4) dst[1] = pack_bf16x2(v[k][2], v[k][3]);
                } else {
                    float* dst = ws.piece_o + (cpiece * G + g) * D + lane * E;
                    if constexpr (E == 4) *reinterpret_cast<float4*>(dst) = make_float4(v[k][0], v[k][1], v[k][2], v[k][3]);
                    else *reinterpret_cast<float2*>(dst) = make_float2(v[k][0], v[k][1]);
                    if (lane == 0) *reinterpret_cast<float2*>(ws.piece_ml + (cpiece * G + g) * 2) = make_float2(Mk[k], dk[k]);
                }
            }
        }
        if (!complete) {
            // ---- level 3: count this CTA's piece; the last one merges all CTA pieces ----------
            Slices sl;
            sl.init(prefix[S], static_cast<int32_t>(gridDim.x), light_ctas, light_units);
            const int32_t c_first = sl.owner(seg_a);
            const int32_t c_last = sl.owner(seg_b - 1);
            const int32_t expected = (U >= C) ? (c_last - c_first + 1) : (seg_b - seg_a);
            __syncwarp();  // the warp's piece stores precede lane 0's release below
            int32_t last = 0;
            if (lane == 0) last = count_piece(ws.counter + seg) == expected - 1;
            last = __shfl_sync(0xffffffffu, last, 0);
            __syncwarp();  // lane 0's acquire precedes every lane's loads of other pieces
            PA_TRACE_STAMP(g_trace, 9);
#ifdef PA_TRACE
            tr_l3 += last ? 2 : 1;
#endif
            if (last) {
                const int64_t row0 = static_cast<int64_t>(s) * Hq + h * G;
                const int32_t first_slot = sl.start(c_first) < seg_a ? 1 : 0;  // the segment's piece in c_first
                merge_pieces<D>(out + row0 * D, first_slot, c_first, c_last, U, C, G, ws, lane, part, row0);
                if (lane == 0) ws.counter[seg] = 0;
                PA_TRACE_STAMP(g_trace, 10);
            }
        }
#ifdef PA_TRACE
        ++tr_groups;
#endif
    }
    PA_TRACE_STAMP(g_trace, 8);
    PA_TRACE_AT(g_trace, 13, tr_groups);
    PA_TRACE_AT(g_trace, 14, tr_l3);
}

template <int D, int NW, int NH, bool APPEND>
cudaError_t launch_impl(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    alignas(64) CUtensorMap tm_k, tm_v;
    // Pool rows of head_dim elements: (block, kv head, token in block).
    const uint64_t rows = static_cast<uint64_t>(a.num_blocks) * a.num_kv_heads * a.block_size;
    cudaError_t e;
    if (D == 128) {
        // (column within a half, pool row, half): one box is a whole 16-row page, stored as
        // two 16 x 128-byte swizzled halves
        e = encode_bf16_3d_sw128(&tm_k, a.k_cache, 64, rows, 2, D * 2, 128, 64, kPageTokens, 2);
        if (e != cudaSuccess) return e;
        e = encode_bf16_3d_sw128(&tm_v, a.v_cache, 64, rows, 2, D * 2, 128, 64, kPageTokens, 2);
    } else {
        e = encode_bf16_2d_sw128(&tm_k, a.k_cache, D, rows, 64, kPageTokens);
        if (e != cudaSuccess) return e;
        e = encode_bf16_2d_sw128(&tm_v, a.v_cache, D, rows, 64, kPageTokens);
    }
    if (e != cudaSuccess) return e;
    const int32_t G = a.num_q_heads / a.num_kv_heads;
    e = cudaFuncSetAttribute(decode_balanced_kernel<D, NW, NH, APPEND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(plan.smem_bytes));
    if (e != cudaSuccess) return e;
    BalWorkspace ws = bal_ws(a.workspace, a.num_seqs, a.num_kv_heads, G, D, plan.num_ctas);
    const WaitDrill drill = wait_drill();

    // Programmatic launch: the grid may be scheduled while the previous kernel in the stream
    // drains; it waits for that kernel (griddepcontrol.wait) before reading any input.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.num_ctas);
    cfg.blockDim = dim3(NW * 32);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_balanced_kernel<D, NW, NH, APPEND>, tm_k, tm_v, static_cast<__nv_bfloat16*>(a.out),
                              static_cast<const __nv_bfloat16*>(a.q), a.block_table, a.max_blocks_per_seq,
                              a.seq_lens, a.num_seqs, a.num_kv_heads, G, a.num_blocks,
                              block_size_log2(a.block_size) - 4, a.scale * kLog2e, plan.stages, plan.stage_bytes, ws,
                              a.err, static_cast<const int4*>(a.k_new), static_cast<const int4*>(a.v_new),
                              a.slot_mapping, static_cast<int4*>(const_cast<void*>(a.k_cache)),
                              static_cast<int4*>(const_cast<void*>(a.v_cache)), a.tables_ready ? 1 : 0,
                              a.pool_ready ? 1 : 0, drill.limit_ns, drill.kind == kDrillDecodeStage ? 1 : 0,
                              a.len_offset, a.part, plan.light_ctas, plan.light_units);
}

// CTAs of the NW-warp kernel that fit on one SM with `smem` bytes of dynamic shared memory
// (checked on the 2-group instantiation, the one with the most registers; 10-warp CTAs exist
// without append only).
template <int D, int NW>
int ctas_per_sm(uint32_t smem) {
    constexpr bool A = NW != 10;
    int n = 0;
    if (cudaFuncSetAttribute(decode_balanced_kernel<D, NW, 2, A>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_balanced_kernel<D, NW, 2, A>, NW * 32, smem) !=
        cudaSuccess)
        return 0;
    return n;
}

}  // namespace

bool plan_decode_balanced(int32_t S, int32_t Hkv, int32_t G, int32_t D, const DeviceInfo& dev, DecodePlan* plan,
                          int32_t max_ctas, bool append) {
    if (G < 4 || G > kBalMaxGroup || (D != 64 && D != 128) || S > kBalMaxSeqs || S < 1) return false;
    const uint32_t stage = bal_stage_bytes(D, G, append);
    // Prefer 8 streaming warps per CTA with as many stages as fit; 4 warps for large groups. A
    // grid capped below the SM count (decode beside another kernel, no append) streams on few
    // SMs, where each warp's page loop sets the rate: there 10 warps come first.
    const bool capped = max_ctas > 0 && max_ctas < dev.num_sms && !append;
    const int order_capped[] = {10, 8, 4}, order_full[] = {8, 4};
    const int* order = capped ? order_capped : order_full;
    const int n_order = capped ? 3 : 2;
    for (int oi = 0; oi < n_order; ++oi) {
        const int NW = order[oi];
        for (int nst = 4; nst >= 2; --nst) {
            const BalLayout L = bal_layout(NW, nst, stage, G, D, S);
            if (L.total > static_cast<uint32_t>(dev.max_smem_optin)) continue;
            int per_sm = 0;
            if (D == 128)
                per_sm = NW == 10 ? ctas_per_sm<128, 10>(L.total)
                                  : NW == 8 ? ctas_per_sm<128, 8>(L.total) : ctas_per_sm<128, 4>(L.total);
            else
                per_sm = NW == 10 ? ctas_per_sm<64, 10>(L.total)
                                  : NW == 8 ? ctas_per_sm<64, 8>(L.total) : ctas_per_sm<64, 4>(L.total);
            if (per_sm < 1) continue;
            plan->path = kDecodeMmaBalanced;
            plan->warps = NW;
            plan->stages = nst;
            plan->stage_bytes = stage;
            plan->smem_bytes = L.total;
            plan->num_ctas = dev.num_sms * per_sm;
            if (max_ctas > 0 && plan->num_ctas > max_ctas) plan->num_ctas = max_ctas;
            // The CTAs that start last (about one in ten) get fewer pages: about as many as
            // an SM streams in the couple of microseconds by which they trail the first ones.
            plan->light_ctas = plan->num_ctas / 10;
            plan->light_units = static_cast<int32_t>(kLightBytes / (2u * kPageTokens * D * 2u));
            plan->workspace_bytes = bal_ws_bytes(S, Hkv, G, D, plan->num_ctas);
            return true;
        }
    }
    return false;
}

namespace {
// 10-warp CTAs serve capped grids without append only (their plan never sets k_new).
template <int D, int NW>
cudaError_t pick_plain(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream, bool wide) {
    if (a.k_new != nullptr) return cudaErrorInvalidValue;
    return wide ? launch_impl<D, NW, 2, false>(a, plan, stream) : launch_impl<D, NW, 1, false>(a, plan, stream);
}

template <int D, int NW>
cudaError_t pick(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream, bool wide) {
    if (a.k_new != nullptr)
        return wide ? launch_impl<D, NW, 2, true>(a, plan, stream) : launch_impl<D, NW, 1, true>(a, plan, stream);
    return wide ? launch_impl<D, NW, 2, false>(a, plan, stream) : launch_impl<D, NW, 1, false>(a, plan, stream);
}
}  // namespace

cudaError_t launch_decode_balanced(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    const bool wide = a.num_q_heads / a.num_kv_heads > 8;  // 9..16 q heads per kv head
    if (a.head_dim == 128) {
        if (plan.warps == 10) return pick_plain<128, 10>(a, plan, stream, wide);
        if (plan.warps == 8) return pick<128, 8>(a, plan, stream, wide);
        return pick<128, 4>(a, plan, stream, wide);
    }
    if (plan.warps == 10) return pick_plain<64, 10>(a, plan, stream, wide);
    if (plan.warps == 8) return pick<64, 8>(a, plan, stream, wide);
    return pick<64, 4>(a, plan, stream, wide);
}

}  // namespace pa

// Test hook: the balanced decode kernel's slices of `units` work units over `ctas` CTAs, as the
// kernel computes them (host copy of the same arithmetic).
extern "C" PA_API pa_status pa_debug_decode_slices(int64_t units, int32_t ctas, int32_t light_ctas, int32_t light_units,
                                                   int64_t* starts, int32_t* owners) {
    if (units < 0 || units > INT32_MAX || ctas < 1 || starts == nullptr) return PA_ERR_INVALID_ARG;
    pa::Slices sl;
    sl.init(units, ctas, light_ctas, light_units);
    for (int32_t c = 0; c <= ctas; ++c) starts[c] = sl.start(c);
    if (owners != nullptr && units > 0)
        for (int64_t u = 0; u < units; ++u) owners[u] = sl.owner(u);
    return PA_OK;
}

#ifdef PA_TRACE
// Profiling builds only: copy the timeline ring to the host / clear it (current device).
extern "C" PA_API int pa_trace_read(void* host, size_t bytes) {
    if (bytes > sizeof(pa::g_trace)) bytes = sizeof(pa::g_trace);
    return static_cast<int>(cudaMemcpyFromSymbol(host, pa::g_trace, bytes));
}
extern "C" PA_API int pa_trace_reset() {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, pa::g_trace);
    if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof(pa::g_trace));
    if (e == cudaSuccess) e = cudaGetSymbolAddress(&p, pa::g_trace_counter);
    if (e == cudaSuccess) e = cudaMemset(p, 0, sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    return static_cast<int>(e);
}
#endif
