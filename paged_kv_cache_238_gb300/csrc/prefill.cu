// Chunked prefill: causal attention of a chunk of new query tokens over the sequence's keys in
// the pool ("vLLM Internals", section 2: long prompts are split into chunks interleaved with
// decode; "vLLM: what PagedAttention turned into", "The scheduler": a chunk is what the token
// budget leaves). Chunk rows are bottom-right aligned: row r of a chunk of C tokens of a
// sequence with L keys sits at position L - C + r and sees keys 0..L - C + r.
//
// Tensor-core kernel (bf16, head_dim 128, GQA group G in {1, 2, 4, 8, 16}). One CTA computes two
// 128-row query tiles (a, b) of one (sequence, kv head): 128/G consecutive chunk tokens times the
// G q heads that share the kv head, so every K/V tile is read once for 2 x 128 rows. Keys go in
// tiles of 128 (eight 16-token blocks gathered through the block table):
//   warp 0     - K producer and warp 10 - V producer: resolve block ids 32 pages ahead and
//                issue 2-D TMA tile copies (128-byte swizzle) of the tile's pages into a 3-stage
//                K ring and a 2-stage V ring, sixteen lanes at once (page x column half); in
//                separate warps so that K never waits for a V stage to be released;
//   warp 1     - owns the tensor memory (512 columns: S and O of each Q tile, fp32; P, bf16,
//                overwrites the first half of its S) and issues, from one elected lane,
//                S = Q K^T (both operands in shared memory) and O += P V (P from tensor
//                memory) as tcgen05.mma kind::f16 (M = N = 128, K = 16 per instruction) in the
//                order PV_a(j), QK_a(j+1), PV_b(j), QK_b(j+1): while one softmax warpgroup works,
//                the tensor core serves the other Q tile;
//   warps 2-5  - softmax of Q tile a, warps 6-9 - of Q tile b: thread = one query row (one
//                TMEM lane); read its S row (twice: max, then exponentials, 64 columns at a
//                time), apply the causal mask on diagonal tiles only, keep the running max and
//                sum in the log2 domain, write P (bf16) into tensor memory, rescale its O row in
//                TMEM only when the max grows by more than 2^8 (the result is exact for any
//                reference value; this only keeps exponentials in range), zero the V rows of
//                keys past the sequence end (their pool cells may hold anything), and finally
//                write O / l.
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
constexpr int kTcRows = 128;        // query rows per Q tile (M)
constexpr int kTcKeys = 128;        // keys per key tile (N of S = Q K^T, K of O += P V)
constexpr int kKWarp = 0;           // K producer
constexpr int kMmaWarp = 1;         // tensor-memory owner and MMA issuer
constexpr int kSoftWarp0 = 2;       // warps 2-5: softmax of Q tile a; warps 6-9: Q tile b
constexpr int kVWarp = 10;          // V producer
constexpr int kTcThreads = 32 * (kVWarp + 1);
constexpr int kLptMaxSeqs = 64;  // sequences ordered longest first inside the kernel
constexpr int kSoftmaxThreads = 256;  // both softmax warpgroups
constexpr uint32_t kHalf = 16384;     // 128 rows x 128 bytes (64 bf16 columns)
constexpr uint32_t kTile = 2 * kHalf; // a 128 x 128 bf16 operand
constexpr float kRescaleThreshold = 8.f;  // log2 units
constexpr int kKStages = 3;           // K ring depth (key tiles in flight)
constexpr int kVStages = 2;           // V ring depth

struct TcSmem {
    static constexpr uint32_t q = 0;                          // Q tiles a, b
    static constexpr uint32_t k = q + 2 * kTile;              // kKStages stages
    static constexpr uint32_t v = k + kKStages * kTile;       // kVStages stages
    static constexpr uint32_t bars = v + kVStages * kTile;
    static constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 9;
    static constexpr uint32_t misc = bars + kNumBars * 8;     // tmem base, abort flag
    static constexpr uint32_t total = misc + 16 + 1024;
};

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* err,
                                              uint64_t limit_ns) {
    if (mbar_wait_bounded(bar, parity, abort, limit_ns)) return true;
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

// Packed fp32 pairs (sm_100 family): one instruction for two lanes' worth of the softmax's
// scale-and-shift and running sums, and a three-input maximum.
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b, float c) {
    uint64_t a, bb, cc, d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %1};" : "=l"(bb) : "f"(b));
    asm("mov.b64 %0, {%1, %1};" : "=l"(cc) : "f"(c));
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(bb), "l"(cc));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(d));
}
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1) {
    uint64_t a, d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(a0), "f"(a1));
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(d0), "f"(d1));
    asm("add.rn.f32x2 %0, %0, %1;" : "+l"(d) : "l"(a));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(d0), "=f"(d1) : "l"(d));
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// 16-byte copy global -> shared (cp.async, L2 only); with `zero` the 16 bytes are zeros and the
// source is not read.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* src, bool zero) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(src),
                 "r"(zero ? 0 : 16)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <int G>
__global__ void __launch_bounds__(kTcThreads, 1) prefill_tc_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ q, const int32_t* __restrict__ block_table,
    int32_t max_blocks, const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ query_start_loc,
    int32_t num_kv_heads, int32_t num_blocks, int32_t sub_log2, float scale_log2, uint32_t* err, uint64_t wait_limit_ns,
    int32_t drill, SharedPrefixPart sp) {
    constexpr int TT = kTcRows / G;  // chunk tokens per Q tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + TcSmem::bars);
    // One barrier phase per use. Key tile j uses K stage j % kKStages and V stage j % kVStages.
    uint64_t* k_full = bars;                       // [kKStages] K tile landed (TMA)
    uint64_t* k_empty = k_full + kKStages;         // [kKStages] the QKs that read the K stage are done
    uint64_t* v_full = k_empty + kKStages;         // [kVStages] V tile landed (TMA)
    uint64_t* v_empty = v_full + kVStages;         // [kVStages] the PVs that read the V stage are done
    uint64_t* s_full = v_empty + kVStages;         // [2] S of Q tile a / b written (commit)
    uint64_t* p_full = s_full + 2;                 // [2] P of Q tile a / b written (4 softmax warps)
    uint64_t* o_done = p_full + 2;                 // [2] last PV of Q tile a / b finished (commit)
    uint64_t* q_full = o_done + 2;                 // Q tiles stored in shared memory (256 threads)
    uint64_t* idle = q_full + 1;                   // every MMA issued has finished (final commit)
    uint64_t* ml_full = idle + 1;                  // shared-prefix mode: both tiles' (max, sum) stored
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + TcSmem::misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + TcSmem::misc + 4);

    const int32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Q tile pairs of one (sequence, kv head) are adjacent in launch order, so they run at the
    // same time and read each K/V tile from L2 after the first of them brings it in. Up to 64
    // sequences go in order of decreasing total length (ties by index): CTA z takes the
    // sequence of rank z, so the longest CTAs start first and the grid ends on short ones.
    __shared__ int32_t lpt_len[kLptMaxSeqs];
    __shared__ int32_t lpt_qsl[kLptMaxSeqs + 1];  // the chunk starts, read with the lengths
    __shared__ int32_t lpt_seq;
    const bool prefix_mode = sp.rows > 0;
    int32_t seq = prefix_mode ? 0 : blockIdx.z;
    const int32_t n_seqs = prefix_mode ? 1 : static_cast<int32_t>(gridDim.z);
    const bool lpt = !prefix_mode && n_seqs <= kLptMaxSeqs;
    if (lpt) {
        if (tid < n_seqs) lpt_len[tid] = __ldg(seq_lens + tid);
        if (tid <= n_seqs) lpt_qsl[tid] = __ldg(query_start_loc + tid);
        __syncthreads();
        if (tid < n_seqs) {
            const int32_t mine = lpt_len[tid];
            int32_t rank = 0;
            for (int32_t u = 0; u < n_seqs; ++u) {
                const int32_t o = lpt_len[u];
                rank += (o > mine || (o == mine && u < tid)) ? 1 : 0;
            }
            if (rank == static_cast<int32_t>(blockIdx.z)) lpt_seq = tid;
        }
        __syncthreads();
        seq = lpt_seq;
    }
    const int32_t h = blockIdx.y;
    const int32_t pair = gridDim.x - 1 - blockIdx.x;  // the longest pairs start first
    const int32_t Hq = G * num_kv_heads;
    // Shared-prefix mode: the "chunk" is one query row per decode sequence (C = sp.rows) and
    // every row sees all L = sp.len prefix keys (no causal bound).
    const int32_t q0 = prefix_mode ? 0 : lpt ? lpt_qsl[seq] : __ldg(query_start_loc + seq);
    const int32_t C = prefix_mode ? sp.rows : (lpt ? lpt_qsl[seq + 1] : __ldg(query_start_loc + seq + 1)) - q0;
    const int32_t L = prefix_mode ? sp.len : lpt ? lpt_len[seq] : __ldg(seq_lens + seq);
    // Shared-prefix mode: one Q tile per CTA, held in both Q slots; its key tiles alternate
    // between the slots (even tiles: a, odd tiles: b), so that both softmax warpgroups and the
    // tensor core's interleaving serve the one tile, and the two parts merge at the end.
    const int32_t t0a = prefix_mode ? pair * TT : 2 * pair * TT, t0b = prefix_mode ? t0a : t0a + TT;
    if (t0a >= C) return;  // uniform over the CTA
    if ((!prefix_mode && C > L) || L > table_tokens(max_blocks, sub_log2) || C < 0) {
        if (tid == 0) raise_error(err, PA_DEVERR_LEN_RANGE);
        return;
    }
    const int32_t P0 = prefix_mode ? L - 1 : L - C;  // position of chunk row 0
    const int32_t n_prefix_tiles = (L + kTcKeys - 1) / kTcKeys;  // shared-prefix mode
    const bool active_b = prefix_mode ? n_prefix_tiles > 1 : t0b < C;
    // key tiles of each slot: those holding keys visible to some row of its Q tile; in
    // shared-prefix mode every prefix tile, split between the slots
    const int32_t n_kv_a = prefix_mode ? (n_prefix_tiles + 1) / 2 : (P0 + min(t0a + TT, C) - 1) / kTcKeys + 1;
    const int32_t n_kv_b = !active_b ? 0 : prefix_mode ? n_prefix_tiles / 2 : (P0 + min(t0b + TT, C) - 1) / kTcKeys + 1;
    // shared-prefix mode: let the next kernel's grid be scheduled now (it waits for this one to
    // complete before it reads anything this kernel writes)
    if (prefix_mode) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int32_t n_kv = prefix_mode ? n_prefix_tiles : max(n_kv_a, n_kv_b);  // key tiles produced
    const int32_t npages = (L + kPageTokens - 1) / kPageTokens;

    // tensor memory columns: S of Q tile x at 128 x (fp32; its P, bf16 pairs, overwrites the
    // first 64 columns once read), O of Q tile x at 256 + 128 x (fp32)
    const bool softmax_warp = warp >= kSoftWarp0 && warp < kVWarp;
    const int32_t xq = softmax_warp ? (warp - kSoftWarp0) >> 2 : 0;  // Q tile of a softmax warp
    const int32_t t0 = xq ? t0b : t0a;
    if (softmax_warp) {
        // ---- Q tiles, by the softmax threads, started before the barriers and the tensor
        // memory are set up: row r = token * G + head, 16-byte copies into the swizzled K-major
        // layout (two 64-column halves); rows past the chunk are zero
        const int32_t ti = tid - 32 * kSoftWarp0 - xq * 128;  // thread within its warpgroup
        uint8_t* sq = smem + TcSmem::q + xq * kTile;
        constexpr int kPer = kTcRows * 16 / 128;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int32_t i = ti + k * 128;
            const int32_t r = i >> 4, c16 = i & 15;  // row, 16-byte chunk of the 256-byte row
            const int32_t t = t0 + r / G, g = r % G;
            const bool in = t < C;
            const __nv_bfloat16* src = in ? q + (static_cast<int64_t>(q0 + t) * Hq + h * G + g) * kTcD + c16 * 8 : q;
            cp_async16(sq + (c16 >> 3) * kHalf + sw128_offset(r, c16 & 7), src, !in);
        }
    }
    // block ids, 32 pages (four key tiles) per window: lane i of a producer warp holds page
    // 32 w + i; the first two windows are fetched before the barriers are set up
    auto page_row = [&](int32_t pg) -> int32_t {
        int32_t phys = 0;  // keys past the sequence end read the null block; masked later
        if (pg < npages) {
            phys = __ldg(block_table + static_cast<int64_t>(seq) * max_blocks + (pg >> sub_log2));
            if (phys < 0 || phys >= num_blocks) {
                raise_error(err, PA_DEVERR_BLOCK_RANGE);
                phys = 0;
            }
        }
        return (((phys * num_kv_heads + h) << sub_log2) + (pg & ((1 << sub_log2) - 1))) * kPageTokens;
    };
    int32_t row_cur = 0, row_nxt = 0;
    if (warp == kKWarp || warp == kVWarp) {
        row_cur = page_row(lane);
        row_nxt = page_row(32 + lane);
    }

    if (tid == 0) {
        *abort_flag = 0;
        for (int i = 0; i < TcSmem::kNumBars; ++i) mbar_init(&bars[i], 1);
        mbar_init(&p_full[0], 4);
        mbar_init(&p_full[1], 4);
        mbar_init(q_full, kSoftmaxThreads);
        mbar_init(ml_full, kSoftmaxThreads);
        fence_mbarrier_init();
    }
    if (warp == kMmaWarp) {
        umma::tmem_alloc(tmem_holder, 512);
        umma::tmem_relinquish();
    }
    umma::fence_before_sync();
    __syncthreads();  // barriers initialised, tensor memory allocated: the producers start now
    umma::fence_after_sync();
    const uint32_t tmem = *tmem_holder;
    if (softmax_warp) {
        cp_async_wait_all();         // this thread's Q copies have landed
        fence_proxy_async_shared();  // before the tensor core reads them
        mbar_arrive(q_full);
    }

    int32_t last_j = -1;  // producers: last key tile whose copies this warp issued
    if (warp == kKWarp || warp == kVWarp) {
        // ============================ producers: K (warp 0), V ===============================
        // Separate warps, so that K copies never wait for a V stage to be freed (V stages
        // are released later, after P V) and run as far ahead as their own ring allows.
        const bool is_v = warp == kVWarp;
        const int32_t nst = is_v ? kVStages : kKStages;
        const void* tm = is_v ? static_cast<const void*>(&tm_v) : static_cast<const void*>(&tm_k);
        uint64_t* full = is_v ? v_full : k_full;
        uint64_t* empty = is_v ? v_empty : k_empty;
        uint8_t* ring = smem + (is_v ? TcSmem::v : TcSmem::k);
        if (lane == 0) prefetch_tensormap(tm);
        // the next window of block ids is fetched while the current one is issued
        int32_t win = 0;
        // With the wait drill on, one CTA's K producer announces 16 bytes more for its first
        // tile than the copies bring: that tile never completes and the MMA warp's wait runs out.
        const uint32_t drill_bytes = (drill && warp == kKWarp && pair == 0 && h == 0 && blockIdx.z == 0) ? 16u : 0u;
        for (int32_t j = 0; j < n_kv; ++j) {
            const int32_t st = j % nst;
            const uint32_t use = static_cast<uint32_t>(j / nst);
            if ((j >> 2) != win) {  // next window of 32 pages
                ++win;
                row_cur = row_nxt;
                row_nxt = page_row(32 * (win + 1) + lane);
            }
            // tile j's stage is free once the MMAs of tile j - nst that read it are done
            bool ok = true;
            if (use > 0 && lane == 0) ok = wait_or_abort(&empty[st], (use - 1) & 1u, abort_flag, err, wait_limit_ns);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            uint8_t* dst = ring + st * kTile;
            if (lane == 0) mbar_arrive_expect_tx(&full[st], kTile + (j == 0 ? drill_bytes : 0u));
            last_j = j;
            const int32_t rk = __shfl_sync(0xffffffffu, row_cur, (j & 3) * 8 + (lane & 7));
            __syncwarp();
            if (lane < 16)  // lane = (column half, page): 16 copies issued at once
                tma_load_2d(dst + (lane >> 3) * kHalf + (lane & 7) * 2048u, tm, (lane >> 3) * 64, rk, &full[st]);
        }
    } else if (warp == kMmaWarp) {
        // ================================ MMA issuer =======================================
        // The whole warp follows the schedule, so every operand stays warp-uniform; one lane,
        // elected once, issues every tcgen05 instruction (a commit tracks only the MMAs of the
        // thread that issues it). Per key tile j the order is
        //   PV_a(j), QK_a(j+1), PV_b(j), QK_b(j+1),
        // so while one softmax warpgroup works on its S, the tensor core serves the other Q
        // tile; a QK may overwrite its S/P columns right after the PV that reads P because
        // MMAs from one thread execute in order.
        const bool leader = umma::elect_one();
        const uint32_t idesc_qk = umma::idesc_bf16_f32(128, 128, 0, 0);  // Q, K both K-major
        const uint32_t idesc_pv = umma::idesc_bf16_f32(128, 128, 0, 1);  // P (TMEM), V MN-major
        // Descriptors are built once and stepped by adding the byte offset / 16 to their
        // start-address field (no carry: every shared address here is below 2^18); building
        // them per instruction costs the single issuing thread more than the MMA itself.
        const uint64_t dq0 = umma::smem_desc_sw128(smem_u32(smem + TcSmem::q), 16, 1024);
        const uint64_t dk0 = umma::smem_desc_sw128(smem_u32(smem + TcSmem::k), 16, 1024);
        const uint64_t dv0 = umma::smem_desc_sw128(smem_u32(smem + TcSmem::v), kHalf, 1024);
        auto qk = [&](int32_t x, int32_t j) {
            const uint64_t dq = dq0 + static_cast<uint64_t>(x) * (kTile >> 4);
            const uint64_t dk = dk0 + static_cast<uint64_t>(j % kKStages) * (kTile >> 4);
            const uint32_t d_s = tmem + x * 128;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint64_t off = ((ks >> 2) * kHalf + (ks & 3) * 32) >> 4;
                if (leader) umma::mma_bf16(d_s, dq + off, dk + off, idesc_qk, ks > 0);
            }
            if (leader) umma::commit(&s_full[x]);
            __syncwarp();
        };
        // O_x += P_x V(j); `acc` false: the first PV of slot x overwrites O_x
        auto pv = [&](int32_t x, int32_t j, bool acc) {
            const uint64_t dv = dv0 + static_cast<uint64_t>(j % kVStages) * (kTile >> 4);
            const uint32_t a_p = tmem + x * 128, d_o = tmem + 256 + x * 128;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {  // 16 keys per instruction: 8 P columns
                if (leader)
                    umma::mma_bf16_tmem_a(d_o, a_p + kk * 8, dv + static_cast<uint64_t>(kk * (2048 >> 4)), idesc_pv,
                                          (acc || kk > 0));
            }
            __syncwarp();
        };
        auto wait_k = [&](int32_t j) {
            const bool ok = wait_or_abort(&k_full[j % kKStages], static_cast<uint32_t>(j / kKStages) & 1u,
                                          abort_flag, err, wait_limit_ns);
            umma::fence_after_sync();
            return ok;
        };
        bool ok = wait_or_abort(q_full, 0, abort_flag, err, wait_limit_ns) && wait_k(0);
        if (prefix_mode) {
            // key tile i: slot i & 1, K and V stages i % kKStages, i % kVStages; per tile
            //   PV_x(i), QK_x(i + 2)
            // so the slots alternate on the tensor core like two Q tiles do
            if (ok) {
                qk(0, 0);
                if (leader) umma::commit(&k_empty[0]);
            }
            if (ok && n_kv > 1) {
                ok = wait_k(1);
                if (ok) {
                    qk(1, 1);
                    if (leader) umma::commit(&k_empty[1 % kKStages]);
                }
            }
            for (int32_t i = 0; i < n_kv && ok; ++i) {
                const int32_t x = i & 1;
                ok = wait_or_abort(&v_full[i % kVStages], static_cast<uint32_t>(i / kVStages) & 1u, abort_flag, err,
                                   wait_limit_ns);
                if (ok) ok = wait_or_abort(&p_full[x], static_cast<uint32_t>(i >> 1) & 1u, abort_flag, err, wait_limit_ns);
                umma::fence_after_sync();
                if (ok) pv(x, i, i >= 2);
                if (ok && leader) {
                    umma::commit(&v_empty[i % kVStages]);
                    if (i + 2 >= n_kv) umma::commit(&o_done[x]);
                }
                if (ok && i + 2 < n_kv) {
                    ok = wait_k(i + 2);
                    if (ok) {
                        qk(x, i + 2);
                        if (leader) umma::commit(&k_empty[(i + 2) % kKStages]);
                    }
                }
                __syncwarp();
            }
        } else if (ok) {
            qk(0, 0);
            if (active_b) qk(1, 0);
            if (leader) umma::commit(&k_empty[0]);
        }
        for (int32_t j = 0; j < n_kv && ok && !prefix_mode; ++j) {
            const bool ua = j < n_kv_a, ub = j < n_kv_b;
            const bool ua1 = j + 1 < n_kv_a, ub1 = j + 1 < n_kv_b;
            ok = wait_or_abort(&v_full[j % kVStages], static_cast<uint32_t>(j / kVStages) & 1u, abort_flag, err, wait_limit_ns);
            if (ok && ua) {
                ok = wait_or_abort(&p_full[0], j & 1, abort_flag, err, wait_limit_ns);  // P_a(j) written, S_a(j) read
                umma::fence_after_sync();
                if (ok) pv(0, j, j > 0);
                if (ok && !ua1 && leader) umma::commit(&o_done[0]);
            }
            if (ok && (ua1 || ub1)) ok = wait_k(j + 1);
            if (ok && ua1) qk(0, j + 1);
            if (ok && ub) {
                ok = wait_or_abort(&p_full[1], j & 1, abort_flag, err, wait_limit_ns);
                umma::fence_after_sync();
                if (ok) pv(1, j, j > 0);
                if (ok && !ub1 && leader) umma::commit(&o_done[1]);
            }
            if (ok && leader) umma::commit(&v_empty[j % kVStages]);
            if (ok && ub1) qk(1, j + 1);
            if (ok && (ua1 || ub1) && leader) umma::commit(&k_empty[(j + 1) % kKStages]);
            __syncwarp();
        }
        if (leader) umma::commit(idle);  // arrives once every MMA issued above has finished
        __syncwarp();
    } else if (softmax_warp) {
        // ================================ softmax warps ===================================
        const int32_t quad = warp & 3;                 // TMEM lane quadrant of this warp
        const int32_t r = quad * 32 + lane;            // query row of this thread
        const int32_t tl = r / G, g = r % G;
        const int32_t n_kv_x = xq ? n_kv_b : n_kv_a;
        const bool row_valid = t0 + tl < C;
        const int32_t pos = min(P0 + t0 + tl, L - 1);  // rows past the chunk: any in-range position
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t tmem_s = tmem + xq * 128, tmem_o = tmem + 256 + xq * 128;
        float m_ref = -INFINITY, l_sum = 0.f;
        bool ok = true;
        for (int32_t j = 0; j < n_kv_x; ++j) {
            ok = wait_or_abort(&s_full[xq], j & 1, abort_flag, err, wait_limit_ns);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            umma::fence_after_sync();
            const int32_t kt = prefix_mode ? 2 * j + xq : j;  // key tile of this step
            const int32_t kbase = kt * kTcKeys;
            const bool diag = kbase + kTcKeys - 1 > pos;  // only these tiles need the causal mask
            // pass 1: row max of the raw scores (scale > 0), eight independent chains
            float mxk[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mxk[k] = -INFINITY;
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                uint32_t raw[2][32];
                umma::ld_32x32b_x32(tmem_s + lane_off + c2 * 64, raw[0]);
                umma::ld_32x32b_x32(tmem_s + lane_off + c2 * 64 + 32, raw[1]);
                umma::wait_ld();
                if (!diag) {
#pragma unroll
                    for (int i = 0; i < 64; i += 2)
                        mxk[(i >> 1) & 7] = max3(mxk[(i >> 1) & 7], __uint_as_float(raw[i >> 5][i & 31]),
                                                 __uint_as_float(raw[i >> 5][(i + 1) & 31]));
                } else {
#pragma unroll
                    for (int i = 0; i < 64; i += 2) {
                        const float x0 = kbase + c2 * 64 + i > pos ? -INFINITY : __uint_as_float(raw[i >> 5][i & 31]);
                        const float x1 =
                            kbase + c2 * 64 + i + 1 > pos ? -INFINITY : __uint_as_float(raw[i >> 5][(i + 1) & 31]);
                        mxk[(i >> 1) & 7] = max3(mxk[(i >> 1) & 7], x0, x1);
                    }
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
            // pass 2: P = 2^(s scale - m) in bf16 pairs over the first 64 columns of S, 32 keys
            // at a time (each group of S columns is read before the P columns that overwrite
            // part of it are written)
            float psk[8];  // four packed pairs of partial sums
#pragma unroll
            for (int k = 0; k < 8; ++k) psk[k] = 0.f;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                uint32_t raw[32];
                umma::ld_32x32b_x32(tmem_s + lane_off + c4 * 32, raw);
                umma::wait_ld();
                if (diag) {  // masked keys: -inf, so their p is exactly 0
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (kbase + c4 * 32 + i > pos) raw[i] = __float_as_uint(-INFINITY);
                }
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float x0, x1;
                    fma2(x0, x1, __uint_as_float(raw[2 * e]), __uint_as_float(raw[2 * e + 1]), scale_log2, neg_m);
                    const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                    add2(psk[2 * (e & 3)], psk[2 * (e & 3) + 1], p0, p1);
                    pk[e] = pack_bf16x2(p0, p1);
                }
                umma::st_32x32b_x16(tmem_s + lane_off + c4 * 16, pk);
            }
            umma::wait_st();
            const float psum = ((psk[0] + psk[1]) + (psk[2] + psk[3])) + ((psk[4] + psk[5]) + (psk[6] + psk[7]));
            l_sum = l_sum * alpha + psum;
            if (!first && grow) {
                // O holds tiles < j under the old reference; the PV of tile j - 1 finished
                // before S of tile j was committed, so O can be rescaled now
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
            // keys of this tile past the sequence end: zero their V rows (thread r: key row r),
            // by the first Q tile that uses key tile kt (the only one in shared-prefix mode)
            if ((prefix_mode || xq == 0 || j >= n_kv_a) && kbase + r >= L) {
                const int32_t st = kt % kVStages;
                const bool okv = wait_or_abort(&v_full[st], static_cast<uint32_t>(kt / kVStages) & 1u, abort_flag, err,
                                               wait_limit_ns);
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
            if (lane == 0) mbar_arrive(&p_full[xq]);
        }
        if (prefix_mode) {
            // Both slots' last PVs have finished once o_done of each has: then every MMA of the
            // CTA has, and the Q slots are free to carry the slots' (max, sum) per row.
            if (ok) ok = wait_or_abort(&o_done[0], 0, abort_flag, err, wait_limit_ns);
            if (ok && active_b) ok = wait_or_abort(&o_done[1], 0, abort_flag, err, wait_limit_ns);
            ok = __all_sync(0xffffffffu, ok);
            float2* mls = reinterpret_cast<float2*>(smem + TcSmem::q);  // [slot][row]
            if (ok) mls[xq * kTcRows + r] = make_float2(m_ref, l_sum);
            mbar_arrive(ml_full);  // every softmax thread, so that no wait below is left hanging
            if (ok) ok = wait_or_abort(ml_full, 0, abort_flag, err, wait_limit_ns);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                // The row's three parts: the prefix keys of slot a and of slot b (unnormalised
                // O_x under max m_x, sum l_x) and its suffix part from the decode grid launched
                // before this kernel (normalised o_s, m_s, l_s), which is waited for here:
                //   M = max(m_a, m_b, m_s),  w_x = 2^(m_x - M),  w_s = l_s 2^(m_s - M)
                //   out = (w_a O_a + w_b O_b + w_s o_s) / (w_a l_a + w_b l_b + w_s)
                // Slot a's warpgroup writes columns 0-63 of the row, slot b's 64-127.
                asm volatile("griddepcontrol.wait;" ::: "memory");
                umma::fence_after_sync();
                const int64_t prow = static_cast<int64_t>(t0 + tl) * Hq + h * G + g;
                const float2 pa = mls[r];
                const float2 pb = active_b ? mls[kTcRows + r] : make_float2(-INFINITY, 0.f);
                float2 ms = make_float2(-INFINITY, 0.f);
                if (row_valid) ms = __ldcg(sp.suffix_ml + prow);
                float M = pa.x;
                if (active_b) M = fmaxf(M, pb.x);
                if (ms.y > 0.f) M = fmaxf(M, ms.x);
                const float wa = fast_exp2(pa.x - M);
                const float wb = active_b ? fast_exp2(pb.x - M) : 0.f;
                const float wsuf = ms.y > 0.f ? ms.y * fast_exp2(ms.x - M) : 0.f;
                const float inv = 1.f / (pa.y * wa + pb.y * wb + wsuf);
                const float ca = wa * inv, cb = wb * inv, cs = wsuf * inv;
                const float* so = sp.suffix_o + prow * kTcD;
                __nv_bfloat16* orow = out + prow * kTcD;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int32_t c = 2 * xq + half;  // 32-column chunk
                    uint32_t ra[32], rb[32];
                    umma::ld_32x32b_x32(tmem + 256 + lane_off + c * 32, ra);
                    if (active_b) umma::ld_32x32b_x32(tmem + 256 + 128 + lane_off + c * 32, rb);
                    umma::wait_ld();
                    if (!active_b) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) rb[i] = 0u;
                    }
                    if (row_valid) {
#pragma unroll
                        for (int v8 = 0; v8 < 4; ++v8) {
                            const float4 s0 = __ldcg(reinterpret_cast<const float4*>(so + c * 32 + v8 * 8));
                            const float4 s1 = __ldcg(reinterpret_cast<const float4*>(so + c * 32 + v8 * 8 + 4));
                            const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
                            float o8[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                o8[e] = fmaf(__uint_as_float(ra[v8 * 8 + e]), ca,
                                             fmaf(__uint_as_float(rb[v8 * 8 + e]), cb, sv[e] * cs));
                            uint4 w;
                            w.x = pack_bf16x2(o8[0], o8[1]);
                            w.y = pack_bf16x2(o8[2], o8[3]);
                            w.z = pack_bf16x2(o8[4], o8[5]);
                            w.w = pack_bf16x2(o8[6], o8[7]);
                            *reinterpret_cast<uint4*>(orow + c * 32 + v8 * 8) = w;
                        }
                    }
                }
            }
        } else if (ok && n_kv_x > 0) {
            ok = wait_or_abort(&o_done[xq], 0, abort_flag, err, wait_limit_ns);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (!prefix_mode && ok && n_kv_x > 0) {
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
    if ((warp == kKWarp || warp == kVWarp) && lane == 0) {
        const int32_t nst = warp == kVWarp ? kVStages : kKStages;
        uint64_t* full = warp == kVWarp ? v_full : k_full;
        for (int32_t j = max(0, last_j - nst + 1); j <= last_j; ++j)
            mbar_wait_timeout(&full[j % nst], static_cast<uint32_t>(j / nst) & 1u, wait_limit_ns);
    }
    if (warp == kMmaWarp && lane == 0) mbar_wait_timeout(idle, 0, wait_limit_ns);  // any thread may wait on the barrier
    umma::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        umma::fence_after_sync();
        umma::tmem_dealloc(tmem, 512);
    }
}

template <int G>
cudaError_t launch_tc(const PrefillArgs& a, cudaStream_t stream) {
    alignas(64) CUtensorMap tm_k, tm_v;
    const uint64_t rows = static_cast<uint64_t>(a.num_blocks) * a.num_kv_heads * a.block_size;
    cudaError_t e = encode_bf16_2d_sw128(&tm_k, a.k_cache, kTcD, rows, 64, kPageTokens);
    if (e != cudaSuccess) return e;
    e = encode_bf16_2d_sw128(&tm_v, a.v_cache, kTcD, rows, 64, kPageTokens);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(prefill_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(TcSmem::total));
    if (e != cudaSuccess) return e;
    constexpr int TT = kTcRows / G;
    const int32_t tiles = (a.max_chunk_len + TT - 1) / TT;
    const int32_t pairs = a.sp.rows > 0 ? tiles : (tiles + 1) / 2;  // Q tiles (pairs) per (sequence, kv head)
    dim3 grid(pairs, a.num_kv_heads, a.sp.rows > 0 ? 1 : a.num_seqs);
    const WaitDrill drill = wait_drill();
    // Shared-prefix mode is a programmatic launch: its CTAs may start while the decode grid
    // before it runs (it waits for that grid before its merge).
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = TcSmem::total;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = a.sp.rows > 0 ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, prefill_tc_kernel<G>, tm_k, tm_v, static_cast<__nv_bfloat16*>(a.out),
                              static_cast<const __nv_bfloat16*>(a.q), a.block_table, a.max_blocks_per_seq, a.seq_lens,
                              a.query_start_loc, a.num_kv_heads, a.num_blocks, block_size_log2(a.block_size) - 4,
                              a.scale * kLog2e, a.err, drill.limit_ns, drill.kind == kDrillPrefillKTile ? 1 : 0, a.sp);
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
    if (a.sp.rows > 0) return cudaErrorInvalidValue;  // shared-prefix mode: tensor-core path only
    const int32_t total_rows = a.num_seqs * a.max_chunk_len;  // upper bound; extra rows exit at once
    return launch_prefill_simt(a, total_rows, stream);
}

}  // namespace pa
