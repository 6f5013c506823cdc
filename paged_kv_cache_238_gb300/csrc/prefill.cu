// Chunked prefill: causal attention of a chunk of new query tokens over the sequence's keys in
// the pool ("vLLM Internals", section 2: long prompts are split into chunks interleaved with
// decode; "vLLM: what PagedAttention turned into", "The scheduler": a chunk is what the token
// budget leaves). Chunk rows are bottom-right aligned: row r of a chunk of C tokens of a
// sequence with L keys sits at position L - C + r and sees keys 0..L - C + r.
//
// Tensor-core kernel (bf16, head_dim 128, GQA group G in {1, 2, 4, 8, 16}). One CTA computes a
// 128-row query tile of one (sequence, kv head): 128/G consecutive chunk tokens times the G q
// heads that share the kv head, so every K/V tile is read once for the whole group. Keys go in
// tiles of 128 (eight 16-token blocks gathered through the block table):
//   warp 0   - producer: resolves block ids 32 pages ahead and issues 2-D TMA tile copies
//              (128-byte swizzle) of the tile's K and V pages into 3-stage rings, sixteen
//              lanes at once (page x column half), since one thread issuing every copy in
//              turn cannot keep up with the tensor cores;
//   warp 1   - owns the tensor memory (512 columns: two S buffers and O in fp32, two P buffers
//              in bf16) and issues, from one thread, S = Q K^T (both operands in shared memory)
//              and O += P V (P from tensor memory) as tcgen05.mma kind::f16 (M = N = 128,
//              K = 16 per instruction), completion tracked with tcgen05.commit on mbarriers;
//              S is double-buffered, so Q K^T of the next key tile overlaps this tile's softmax;
//   warps 2-5- softmax: thread = one query row (one TMEM lane); reads its S row, applies the
//              causal mask, keeps the running max and sum in the log2 domain, writes P (bf16)
//              into tensor memory for the second MMA, rescales its O row in TMEM only
//              when the max grows by more than 2^8 (the result is exact for any reference
//              value; this only keeps exponentials in range), zeroes the V rows of keys past
//              the sequence end (their pool cells may hold anything), and finally writes O / l.
// Every wait is bounded; a timeout sets PA_DEVERR_WAIT_TIMEOUT and the CTA winds down.
#include <cuda.h>
#include <math.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kTcD = 128;
constexpr int kTcRows = 128;       // query rows per tile (M)
constexpr int kTcKeys = 128;       // keys per tile (N of S = Q K^T, K of O += P V)
constexpr int kTcThreads = 224;    // K producer, MMA warp, 4 softmax warps, V producer
constexpr int kSoftmaxThreads = 128;  // warps 2-5
constexpr int kVWarp = 6;
constexpr uint32_t kHalf = 16384;  // 128 rows x 128 bytes (64 bf16 columns)
constexpr uint32_t kTile = 2 * kHalf;  // a 128 x 128 bf16 operand
constexpr float kRescaleThreshold = 8.f;  // log2 units
constexpr int kTcStages = 3;             // K and V ring depth (key tiles in flight)

struct TcSmem {
    static constexpr uint32_t q = 0;
    static constexpr uint32_t k = q + kTile;                 // kTcStages stages
    static constexpr uint32_t v = k + kTcStages * kTile;     // kTcStages stages
    static constexpr uint32_t bars = v + kTcStages * kTile;
    static constexpr int kNumBars = 4 * kTcStages + 8;
    static constexpr uint32_t misc = bars + kNumBars * 8;  // tmem base, abort flag
    static constexpr uint32_t total = misc + 16 + 1024;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* err) {
    if (mbar_wait_bounded(bar, parity, abort)) return true;
    if (!*abort) raise_error(err, PA_DEVERR_WAIT_TIMEOUT);
    *abort = 1;
    return false;
}

// 2^x with the hardware approximation (relative error about 2^-22; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int G>
__global__ void __launch_bounds__(kTcThreads, 1) prefill_tc_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ block_table,
    int32_t max_blocks, const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ query_start_loc,
    int32_t num_kv_heads, int32_t num_blocks, float scale_log2, uint32_t* err) {
    constexpr int TT = kTcRows / G;  // chunk tokens per tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + TcSmem::bars);
    // K/V stage st serves key tiles j with j % kTcStages == st; S, P and PV buffers b serve
    // tiles with j % 2 == b; one barrier phase per use
    uint64_t* k_full = bars;                       // [stages] K tile landed (TMA)
    uint64_t* k_empty = k_full + kTcStages;        // [stages] QK done with the K stage (commit)
    uint64_t* v_full = k_empty + kTcStages;        // [stages] V tile landed (TMA)
    uint64_t* v_empty = v_full + kTcStages;        // [stages] PV done with the V stage (commit)
    uint64_t* s_full = v_empty + kTcStages;        // [2] S buffer written (commit)
    uint64_t* p_full = s_full + 2;                 // [2] P written to TMEM, S read (4 softmax warps)
    uint64_t* pv_done = p_full + 2;                // [2] PV of the tile finished (commit)
    uint64_t* idle = pv_done + 2;                  // every MMA issued has finished (final commit)
    uint64_t* q_full = idle + 1;                   // Q tile stored in shared memory (128 softmax threads)
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + TcSmem::misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + TcSmem::misc + 4);

    const int32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Query tiles of one (sequence, kv head) are adjacent in launch order, so they run at the
    // same time and read each K/V tile from L2 after the first of them brings it in.
    const int32_t seq = blockIdx.z, h = blockIdx.y;
    const int32_t tile = gridDim.x - 1 - blockIdx.x;  // the longest tiles start first
    const int32_t Hq = G * num_kv_heads;
    const int32_t q0 = __ldg(query_start_loc + seq);
    const int32_t C = __ldg(query_start_loc + seq + 1) - q0;
    const int32_t L = __ldg(seq_lens + seq);
    const int32_t t0 = tile * TT;
    if (t0 >= C) return;  // uniform over the CTA
    if (C > L || L > max_blocks * kBlock || C < 0) {
        if (tid == 0) raise_error(err, PA_DEVERR_LEN_RANGE);
        return;
    }
    const int32_t P0 = L - C;                             // position of chunk row 0
    const int32_t t_end = min(t0 + TT, C);
    const int32_t max_pos = P0 + t_end - 1;
    const int32_t n_kv = max_pos / kTcKeys + 1;           // key tiles that hold visible keys
    const int32_t npages = (L + kBlock - 1) / kBlock;

    if (tid == 0) {
        *abort_flag = 0;
        for (int i = 0; i < TcSmem::kNumBars; ++i) mbar_init(&bars[i], 1);
        mbar_init(&p_full[0], 4);
        mbar_init(&p_full[1], 4);
        mbar_init(q_full, kSoftmaxThreads);
        fence_mbarrier_init();
    }
    if (warp == 1) {
        umma::tmem_alloc(tmem_holder, 512);
        umma::tmem_relinquish();
    }
    umma::fence_before_sync();
    __syncthreads();  // barriers initialised, tensor memory allocated: the producer starts now
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_holder;
    if (warp >= 2 && warp < kVWarp) {
        // ---- Q tile, by the softmax threads while the first K/V copies are in flight: row
        // r = token * G + head, 16-byte loads (all issued before any store) into the swizzled
        // K-major layout (two 64-column halves); rows past the chunk are zero
        constexpr int kPer = kTcRows * 16 / kSoftmaxThreads;
        int4 v[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int32_t i = (tid - 64) + k * kSoftmaxThreads;
            const int32_t r = i >> 4, c16 = i & 15;  // row, 16-byte chunk of the 256-byte row
            const int32_t t = t0 + r / G, g = r % G;
            v[k] = make_int4(0, 0, 0, 0);
            if (t < C) v[k] = *reinterpret_cast<const int4*>(q + (static_cast<int64_t>(q0 + t) * Hq + h * G + g) * kTcD + c16 * 8);
        }
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int32_t i = (tid - 64) + k * kSoftmaxThreads;
            const int32_t r = i >> 4, c16 = i & 15;
            *reinterpret_cast<int4*>(smem + TcSmem::q + (c16 >> 3) * kHalf + sw128_offset(r, c16 & 7)) = v[k];
        }
        fence_proxy_async_shared();  // generic stores before the tensor core reads them
        mbar_arrive(q_full);
    }
    // tensor memory columns: S buffers at 0 and 128 (fp32), O at 256 (fp32), P buffers at 384
    // and 448 (bf16 pairs)
    const uint32_t tmem_o = tmem + 256, tmem_p = tmem + 384;

    int32_t last_j = -1;  // producers: last key tile whose copies this warp issued
    if (warp == 0 || warp == kVWarp) {
        // ============================ producers: K (warp 0), V ===============================
        // Separate warps, so that K copies never wait for a V stage to be freed (V stages
        // are released later, after P V) and run as far ahead as their own ring allows.
        const bool is_v = warp == kVWarp;
        const void* tm = is_v ? static_cast<const void*>(&tm_v) : static_cast<const void*>(&tm_k);
        uint64_t* full = is_v ? v_full : k_full;
        uint64_t* empty = is_v ? v_empty : k_empty;
        uint8_t* ring = smem + (is_v ? TcSmem::v : TcSmem::k);
        if (lane == 0) prefetch_tensormap(tm);
        // block ids, 32 pages (four key tiles) per window: lane i holds page 32 w + i; the
        // next window is fetched while the current one is issued
        auto page_row = [&](int32_t pg) -> int32_t {
            int32_t phys = 0;  // keys past the sequence end read the null block; masked later
            if (pg < npages) {
                phys = __ldg(block_table + static_cast<int64_t>(seq) * max_blocks + pg);
                if (phys < 0 || phys >= num_blocks) {
                    raise_error(err, PA_DEVERR_BLOCK_RANGE);
                    phys = 0;
                }
            }
            return (phys * num_kv_heads + h) * kBlock;
        };
        int32_t win = 0;
        int32_t row_cur = page_row(lane), row_nxt = page_row(32 + lane);
        for (int32_t j = 0; j < n_kv; ++j) {
            const int32_t st = j % kTcStages;
            const uint32_t use = static_cast<uint32_t>(j / kTcStages);
            if ((j >> 2) != win) {  // next window of 32 pages
                ++win;
                row_cur = row_nxt;
                row_nxt = page_row(32 * (win + 1) + lane);
            }
            // tile j's stage is free once the MMA of tile j - stages that read it is done
            bool ok = true;
            if (use > 0 && lane == 0) ok = wait_or_abort(&empty[st], (use - 1) & 1u, abort_flag, err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            uint8_t* dst = ring + st * kTile;
            if (lane == 0) mbar_arrive_expect_tx(&full[st], kTile);
            last_j = j;
            const int32_t rk = __shfl_sync(0xffffffffu, row_cur, (j & 3) * 8 + (lane & 7));
            __syncwarp();
            if (lane < 16)  // lane = (column half, page): 16 copies issued at once
                tma_load_2d(dst + (lane >> 3) * kHalf + (lane & 7) * 2048u, tm, (lane >> 3) * 64, rk, &full[st]);
        }
    } else if (warp == 1) {
        // ================================ MMA issuer =======================================
        // The whole warp follows the schedule, so every operand stays warp-uniform; one lane,
        // elected once, issues every tcgen05 instruction (a commit tracks only the MMAs of the
        // thread that issues it).
        {
            const bool leader = umma::elect_one();
            const uint32_t idesc_qk = umma::idesc_bf16_f32(128, 128, 0, 0);  // Q, K both K-major
            const uint32_t idesc_pv = umma::idesc_bf16_f32(128, 128, 0, 1);  // P (TMEM), V MN-major
            // Descriptors are built once and stepped by adding the byte offset / 16 to their
            // start-address field (no carry: every shared address here is below 2^18); building
            // them per instruction costs the single issuing thread more than the MMA itself.
            const uint64_t dq = umma::smem_desc_sw128(smem_u32(smem + TcSmem::q), 16, 1024);
            const uint64_t dk0 = umma::smem_desc_sw128(smem_u32(smem + TcSmem::k), 16, 1024);
            const uint64_t dv0 = umma::smem_desc_sw128(smem_u32(smem + TcSmem::v), kHalf, 1024);
            auto issue_qk = [&](int32_t j) -> bool {
                const int32_t b = j & 1, st = j % kTcStages;
                if (!wait_or_abort(&k_full[st], static_cast<uint32_t>(j / kTcStages) & 1u, abort_flag, err)) return false;
                umma::fence_after_sync();
                const uint64_t dk = dk0 + static_cast<uint64_t>(st) * (kTile >> 4);
                const uint32_t d_s = tmem + b * 128;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t off = ((ks >> 2) * kHalf + (ks & 3) * 32) >> 4;
                    if (leader) umma::mma_bf16(d_s, dq + off, dk + off, idesc_qk, ks > 0);
                }
                if (leader) {
                    umma::commit(&s_full[b]);
                    umma::commit(&k_empty[st]);
                }
                __syncwarp();
                return true;
            };
            bool ok = wait_or_abort(q_full, 0, abort_flag, err);
            if (ok) ok = issue_qk(0);
            if (ok && n_kv > 1) ok = issue_qk(1);
            for (int32_t j = 0; j < n_kv && ok; ++j) {
                const int32_t b = j & 1, st = j % kTcStages;
                ok = wait_or_abort(&p_full[b], (j >> 1) & 1, abort_flag, err);   // P_j written, S_j read
                if (ok) ok = wait_or_abort(&v_full[st], static_cast<uint32_t>(j / kTcStages) & 1u, abort_flag, err);
                if (!ok) break;
                umma::fence_after_sync();
                const uint64_t dv = dv0 + static_cast<uint64_t>(st) * (kTile >> 4);
                const uint32_t a_p = tmem_p + b * 64;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {  // 16 keys per instruction: 8 P columns
                    if (leader)
                        umma::mma_bf16_tmem_a(tmem_o, a_p + kk * 8, dv + static_cast<uint64_t>(kk * (2048 >> 4)),
                                              idesc_pv, (j > 0 || kk > 0));
                }
                if (leader) {
                    umma::commit(&pv_done[b]);
                    umma::commit(&v_empty[st]);
                }
                __syncwarp();
                if (j + 2 < n_kv) ok = issue_qk(j + 2);
            }
            if (leader) umma::commit(idle);  // arrives once every MMA issued above has finished
            __syncwarp();
        }
    } else if (warp < kVWarp) {
        // ================================ softmax warps ===================================
        const int32_t quad = warp & 3;                 // TMEM lane quadrant of this warp
        const int32_t r = quad * 32 + lane;            // query row of this thread
        const int32_t tl = r / G, g = r % G;
        const bool row_valid = t0 + tl < C;
        const int32_t pos = min(P0 + t0 + tl, L - 1);  // rows past the chunk: any in-range position
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        float m_ref = -INFINITY, l_sum = 0.f;
        bool ok = true;
        for (int32_t j = 0; j < n_kv; ++j) {
            const int32_t b = j & 1;
            ok = wait_or_abort(&s_full[b], (j >> 1) & 1, abort_flag, err);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            umma::fence_after_sync();
            const int32_t kbase = j * kTcKeys;
            float sv[128];
            {
                uint32_t raw[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) umma::ld_32x32b_x32(tmem + b * 128 + lane_off + c * 32, raw[c]);
                umma::wait_ld();
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) sv[c * 32 + i] = __uint_as_float(raw[c][i]);
            }
            // row max of the raw scores (scale > 0), eight independent chains; only the tiles
            // that cross this row's diagonal need the causal mask
            float mxk[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mxk[k] = -INFINITY;
            if (kbase + kTcKeys - 1 <= pos) {
#pragma unroll
                for (int i = 0; i < 128; ++i) mxk[i & 7] = fmaxf(mxk[i & 7], sv[i]);
            } else {
#pragma unroll
                for (int i = 0; i < 128; ++i) {
                    const float x = (kbase + i <= pos) ? sv[i] : -INFINITY;
                    sv[i] = x;
                    mxk[i & 7] = fmaxf(mxk[i & 7], x);
                }
            }
            const float mx = fmaxf(fmaxf(fmaxf(mxk[0], mxk[1]), fmaxf(mxk[2], mxk[3])),
                                   fmaxf(fmaxf(mxk[4], mxk[5]), fmaxf(mxk[6], mxk[7]))) *
                             scale_log2;
            // reference max: move it only when the tile max exceeds it by more than 2^8
            const bool first = (j == 0);
            const bool grow = first || (mx > m_ref + kRescaleThreshold);
            const float m_new = grow ? fmaxf(m_ref, mx) : m_ref;
            const float alpha = first ? 0.f : fast_exp2(m_ref - m_new);
            const float neg_m = -m_new;
            // the P columns of tile j served PV of tile j - 2
            if (j >= 2) {
                const bool okp = wait_or_abort(&pv_done[b], ((j >> 1) - 1) & 1, abort_flag, err);
                if (!__all_sync(0xffffffffu, okp)) {
                    ok = false;
                    break;
                }
            }
            float psk[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) psk[k] = 0.f;
#pragma unroll
            for (int half = 0; half < 2; ++half) {  // 64 keys -> 32 columns of bf16 pairs
                uint32_t pk[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const float p0 = fast_exp2(fmaf(sv[half * 64 + 2 * e], scale_log2, neg_m));
                    const float p1 = fast_exp2(fmaf(sv[half * 64 + 2 * e + 1], scale_log2, neg_m));
                    psk[(2 * e) & 7] += p0;
                    psk[(2 * e + 1) & 7] += p1;
                    pk[e] = pack_bf16x2(p0, p1);
                }
                umma::st_32x32b_x32(tmem_p + b * 64 + lane_off + half * 32, pk);
            }
            umma::wait_st();
            const float psum = ((psk[0] + psk[1]) + (psk[2] + psk[3])) + ((psk[4] + psk[5]) + (psk[6] + psk[7]));
            l_sum = l_sum * alpha + psum;
            if (!first && grow) {
                // O holds tiles < j under the old reference: wait for PV of tile j - 1, rescale
                const bool oko = wait_or_abort(&pv_done[b ^ 1], ((j - 1) >> 1) & 1, abort_flag, err);
                if (!__all_sync(0xffffffffu, oko)) {
                    ok = false;
                    break;
                }
                umma::fence_after_sync();
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t raw[32];
                    umma::ld_32x32b_x32(tmem_o + lane_off + c * 32, raw);
                    umma::wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) raw[i] = __float_as_uint(__uint_as_float(raw[i]) * alpha);
                    umma::st_32x32b_x32(tmem_o + lane_off + c * 32, raw);
                }
                umma::wait_st();
            }
            m_ref = m_new;
            // keys of this tile past the sequence end: zero their V rows (thread r: key row r)
            if (kbase + r >= L) {
                const int32_t st = j % kTcStages;
                const bool okv = wait_or_abort(&v_full[st], static_cast<uint32_t>(j / kTcStages) & 1u, abort_flag, err);
                if (okv) {
                    uint8_t* sv_tile = smem + TcSmem::v + st * kTile;
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            *reinterpret_cast<int4*>(sv_tile + hf * kHalf + r * 128u + c * 16u) = make_int4(0, 0, 0, 0);
                }
            }
            fence_proxy_async_shared();
            umma::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[b]);
        }
        if (ok) {
            ok = wait_or_abort(&pv_done[(n_kv - 1) & 1], ((n_kv - 1) >> 1) & 1, abort_flag, err);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (ok) {
            umma::fence_after_sync();
            const float inv = 1.f / l_sum;
            __nv_bfloat16* orow = out + (static_cast<int64_t>(q0 + t0 + tl) * Hq + h * G + g) * kTcD;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t raw[32];
                umma::ld_32x32b_x32(tmem_o + lane_off + c * 32, raw);
                umma::wait_ld();
                if (row_valid) {
#pragma unroll
                    for (int v4 = 0; v4 < 4; ++v4) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(raw[v4 * 8 + 0]) * inv, __uint_as_float(raw[v4 * 8 + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(raw[v4 * 8 + 2]) * inv, __uint_as_float(raw[v4 * 8 + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(raw[v4 * 8 + 4]) * inv, __uint_as_float(raw[v4 * 8 + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(raw[v4 * 8 + 6]) * inv, __uint_as_float(raw[v4 * 8 + 7]) * inv);
                        *reinterpret_cast<uint4*>(orow + c * 32 + v4 * 8) = w;
                    }
                }
            }
        }
    }

    // ---- wind down: copies landed and MMAs retired before shared and tensor memory go ------
    if ((warp == 0 || warp == kVWarp) && lane == 0) {
        uint64_t* full = warp == kVWarp ? v_full : k_full;
        for (int32_t j = max(0, last_j - kTcStages + 1); j <= last_j; ++j)
            mbar_wait_timeout(&full[j % kTcStages], static_cast<uint32_t>(j / kTcStages) & 1u);
    }
    if (warp == 1 && lane == 0) mbar_wait_timeout(idle, 0);  // any thread may wait on the barrier
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        umma::fence_after_sync();
        umma::tmem_dealloc(tmem, 512);
    }
}

template <int G>
cudaError_t launch_tc(const PrefillArgs& a, cudaStream_t stream) {
    alignas(64) CUtensorMap tm_k, tm_v;
    const uint64_t rows = static_cast<uint64_t>(a.num_blocks) * a.num_kv_heads * kBlock;
    cudaError_t e = encode_bf16_2d_sw128(&tm_k, a.k_cache, kTcD, rows, 64, kBlock);
    if (e != cudaSuccess) return e;
    e = encode_bf16_2d_sw128(&tm_v, a.v_cache, kTcD, rows, 64, kBlock);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(prefill_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(TcSmem::total));
    if (e != cudaSuccess) return e;
    constexpr int TT = kTcRows / G;
    const int32_t tiles = (a.max_chunk_len + TT - 1) / TT;
    dim3 grid(tiles, a.num_kv_heads, a.num_seqs);
    prefill_tc_kernel<G><<<grid, kTcThreads, TcSmem::total, stream>>>(
        tm_k, tm_v, static_cast<__nv_bfloat16*>(a.out), static_cast<const __nv_bfloat16*>(a.q), a.block_table,
        a.max_blocks_per_seq, a.seq_lens, a.query_start_loc, a.num_kv_heads, a.num_blocks, a.scale * kLog2e, a.err);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
    const int32_t G = a.num_q_heads / a.num_kv_heads;
    const bool tc = a.dtype == PA_BF16 && a.head_dim == kTcD && (G == 1 || G == 2 || G == 4 || G == 8 || G == 16) &&
                    a.num_kv_heads <= 65535 && a.num_seqs <= 65535 &&
                    static_cast<int>(TcSmem::total) <= dev.max_smem_optin;
    if (tc) {
        switch (G) {
            case 1: return launch_tc<1>(a, stream);
            case 2: return launch_tc<2>(a, stream);
            case 4: return launch_tc<4>(a, stream);
            case 8: return launch_tc<8>(a, stream);
            default: return launch_tc<16>(a, stream);
        }
    }
    const int32_t total_rows = a.num_seqs * a.max_chunk_len;  // upper bound; extra rows exit at once
    return launch_prefill_simt(a, total_rows, stream);
}

}  // namespace pa
