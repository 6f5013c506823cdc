/*
 * Paged-KV attention oracle: plain, slow, obviously correct CPU code in fp64.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or load
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark do. It shares no code, header or constant with the CUDA library.
 *
 * What it computes (sources are the three web pages on vLLM's paged KV cache):
 *  - KV lives in fixed-size physical blocks placed anywhere in memory; a block
 *    table maps a sequence's logical block i to a physical block
 *    ("vLLM Internals", section 1.1; "My Understanding of vLLM and
 *    PagedAttention", sections "Logical Blocks", "Physical Blocks",
 *    "Block Table").
 *  - The block size is 16 tokens by default ("vLLM: what PagedAttention turned
 *    into", intro table and "The problem PagedAttention was actually solving");
 *    the same page reports that sizes from 16 to 128 perform alike, so the block
 *    size is an argument (bs below).
 *  - A slot is an int64 index into the pool, one per new token, used to write
 *    new K/V ("vLLM: what PagedAttention turned into", same section: the int64
 *    slot_mapping mirrored to the device).
 *  - Attention gathers the scattered blocks back into logical token order and
 *    computes ordinary attention ("My Understanding...", "PagedAttention CUDA
 *    Kernel" and "Step 4 - Attention Computation"). Paging only relocates K/V,
 *    so the exact result is softmax(scale * q K^T) V over the visible keys.
 *
 * Readings taken where the pages are silent:
 *  - Pool layout: separate K and V arrays, each [num_blocks][H_kv][bs][D].
 *  - slot = physical_block * bs + offset; positions are 0-based, so position p
 *    lives in logical block p / bs at offset p % bs.
 *  - A negative slot means "no write" (the token is skipped).
 *  - GQA: query head h reads kv head h / (H_q / H_kv).
 *  - seq_len counts every key of the sequence, including the current token.
 *  - Chunked prefill is bottom-right aligned: chunk row r of a sequence with
 *    total length L and chunk length C sits at position L - C + r and sees
 *    keys 0..L - C + r.
 *  - A sequence of length 0 (decode) produces an all-zero output row.
 *
 * Parity pins (checked by the CPU tests): brute-force attention on contiguous
 * K/V, a library attention routine, closed forms, permutation invariance of
 * physical ids, alias-versus-copy of shared prefix blocks, null-block
 * poisoning, and the page's worked block-table example.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif


enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };
enum { ORACLE_OK = 0, ORACLE_ERR = 1 };

/* Read element i of a stored array as fp64. bf16 is the upper half of an
 * IEEE binary32, so widening is exact. */
static double load_elem(const void* base, size_t i, int dtype) {
    if (dtype == ORACLE_F32) {
        return (double)((const float*)base)[i];
    }
    uint32_t bits = ((uint32_t)((const uint16_t*)base)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * Write the K/V rows of T new tokens into their slots. Token t goes to
 * physical block slot[t] / bs at in-block offset slot[t] % bs (bs = block_size,
 * 16 by default; "vLLM: what PagedAttention turned into" gives 16 and says
 * 16-128 perform alike), for every kv head. The copy is bitwise in the stored
 * element type (elem_bytes 4 or 2).
 * Returns ORACLE_ERR (and writes nothing more) on a slot beyond the pool.
 */
int oracle_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, int32_t T, int32_t H_kv, int32_t D,
                             int32_t num_blocks, int32_t block_size, int32_t elem_bytes) {
    const size_t row = (size_t)D * (size_t)elem_bytes;
    if (block_size <= 0) return ORACLE_ERR;
    for (int32_t t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        if (block >= num_blocks) return ORACLE_ERR;
        for (int32_t h = 0; h < H_kv; ++h) {
            size_t src = ((size_t)t * H_kv + h) * row;
            size_t dst = (((size_t)block * H_kv + h) * (size_t)block_size + (size_t)offset) * row;
            memcpy((char*)k_cache + dst, (const char*)k + src, row);
            memcpy((char*)v_cache + dst, (const char*)v + src, row);
        }
    }
    return ORACLE_OK;
}

/*
 * Attention over the paged pool, fp64 throughout.
 *
 * out            [T_q][H_q][D] fp64, T_q = S (decode) or query_start_loc[S] (prefill)
 * q              [T_q][H_q][D] in the stored dtype
 * k_cache/v_cache [num_blocks][H_kv][block_size][D] in the stored dtype
 * block_table    [S][max_blocks_per_seq] int32
 * seq_lens       [S] total keys per sequence, current token(s) included
 * query_start_loc NULL for decode (one query row per sequence, at position
 *                len - 1); otherwise [S + 1] prefix sums of chunk lengths.
 */
int oracle_attention(double* out, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_table, int32_t max_blocks_per_seq,
                     const int32_t* seq_lens, const int32_t* query_start_loc, int32_t S,
                     int32_t H_q, int32_t H_kv, int32_t D, int32_t num_blocks, int32_t block_size,
                     double scale, int32_t dtype, int32_t num_threads) {
    if (S < 0 || H_q <= 0 || H_kv <= 0 || D <= 0 || H_q % H_kv != 0 || block_size <= 0) return ORACLE_ERR;
    const int32_t group = H_q / H_kv;

    /* Validate the tables first so the parallel loop below cannot fail. */
    for (int32_t i = 0; i < S; ++i) {
        int32_t len = seq_lens[i];
        if (len < 0) return ORACLE_ERR;
        int32_t n_blocks = (len + block_size - 1) / block_size;
        if (n_blocks > max_blocks_per_seq) return ORACLE_ERR;
        for (int32_t j = 0; j < n_blocks; ++j) {
            int32_t phys = block_table[(size_t)i * max_blocks_per_seq + j];
            if (phys < 0 || phys >= num_blocks) return ORACLE_ERR;
        }
        if (query_start_loc) {
            int32_t chunk = query_start_loc[i + 1] - query_start_loc[i];
            if (chunk < 0 || chunk > len) return ORACLE_ERR;
        }
    }

#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif

    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int32_t i = 0; i < S; ++i) {
        const int32_t len = seq_lens[i];
        const int32_t chunk = query_start_loc ? query_start_loc[i + 1] - query_start_loc[i] : 1;
        const int32_t row0 = query_start_loc ? query_start_loc[i] : i;

        if (len == 0) {
            /* Only reachable for decode (a prefill chunk cannot exceed len). */
            memset(out + (size_t)row0 * H_q * D, 0, sizeof(double) * (size_t)H_q * D);
            continue;
        }

        /* Gather: logical token j of kv head g comes from physical block
         * block_table[i][j / bs] at offset j % bs. */
        double* K = (double*)malloc(sizeof(double) * (size_t)H_kv * len * D);
        double* V = (double*)malloc(sizeof(double) * (size_t)H_kv * len * D);
        double* z = (double*)malloc(sizeof(double) * (size_t)len);
        double* qd = (double*)malloc(sizeof(double) * (size_t)D);
        if (!K || !V || !z || !qd) {
            free(K); free(V); free(z); free(qd);
            failed = 1;
            continue;
        }
        for (int32_t g = 0; g < H_kv; ++g) {
            for (int32_t j = 0; j < len; ++j) {
                int32_t phys = block_table[(size_t)i * max_blocks_per_seq + j / block_size];
                size_t src = (((size_t)phys * H_kv + g) * (size_t)block_size + (size_t)(j % block_size)) * D;
                size_t dst = ((size_t)g * len + j) * D;
                for (int32_t d = 0; d < D; ++d) {
                    K[dst + d] = load_elem(k_cache, src + d, dtype);
                    V[dst + d] = load_elem(v_cache, src + d, dtype);
                }
            }
        }

        for (int32_t r = 0; r < chunk; ++r) {
            const int32_t pos = len - chunk + r; /* keys 0..pos are visible */
            const size_t qrow = (size_t)(row0 + r) * H_q;
            for (int32_t h = 0; h < H_q; ++h) {
                const int32_t g = h / group;
                const double* Kg = K + (size_t)g * len * D;
                const double* Vg = V + (size_t)g * len * D;
                const size_t qoff = (qrow + h) * D;
                for (int32_t d = 0; d < D; ++d) qd[d] = load_elem(q, qoff + d, dtype);

                double zmax = -INFINITY;
                for (int32_t j = 0; j <= pos; ++j) {
                    double dot = 0.0;
                    for (int32_t d = 0; d < D; ++d) dot += qd[d] * Kg[(size_t)j * D + d];
                    z[j] = scale * dot;
                    if (z[j] > zmax) zmax = z[j];
                }
                double denom = 0.0;
                for (int32_t j = 0; j <= pos; ++j) {
                    z[j] = exp(z[j] - zmax);
                    denom += z[j];
                }
                double* o = out + (qrow + h) * D;
                for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
                for (int32_t j = 0; j <= pos; ++j) {
                    const double w = z[j] / denom;
                    for (int32_t d = 0; d < D; ++d) o[d] += w * Vg[(size_t)j * D + d];
                }
            }
        }
        free(K);
        free(V);
        free(z);
        free(qd);
    }
    return failed ? ORACLE_ERR : ORACLE_OK;
}
