// Host-side block manager for the paged KV pool: which physical blocks (16 tokens by default;
// 32, 64 or 128 through pa_bm_create_bs) a request owns, which freed blocks still hold reusable prefixes, and the block table / slot mapping
// the kernels read.
//
// Model ("vLLM: what PagedAttention turned into", "The block pool, and the two tricks in it"
// and "What a block hash actually is"; "vLLM Internals", section 1.2):
//  * The pool's blocks sit in one free queue, an intrusive doubly linked list over the block
//    records with sentinel head and tail, so a block leaves it from anywhere in O(1) and no
//    allocation happens while it is edited. The first block taken at construction is the null
//    block: an ordinary id meaning "no block", never handed out.
//  * A freed block without a hash can never be hit again and goes to the front (reused first);
//    a freed block with a hash goes to the back (evicted last). A request's blocks are freed
//    tail first, so a prefix's tail is offered for eviction before its parents.
//  * Freed blocks keep their hash and stay in the cache map; a block is evicted from the map
//    only when it is taken from the queue for new content.
//  * A block hash is SHA-256(parent hash || the block's token ids as int32 little-endian ||
//    extra key bytes), chained from SHA-256(seed); a per-request salt enters the first block
//    only; the cache key appends the group id (4 bytes, big-endian). Prefix lookup takes the
//    longest run of cached full blocks and stops at the first miss; a prompt never hits in
//    full (at most (len - 1) / block_size blocks come from the cache).
//  * Blocks are reference counted: a forked request shares every block, and appending into a
//    shared, partly filled last block first moves the request to a private copy
//    (copy-on-write); the (source, destination) pairs wait for pa_copy_blocks.
//  * A full block enters the cache when the caller commits that its K/V has been computed; a
//    key already cached keeps its block and the new block stays unhashed.
#include <array>
#include <cstdint>
#include <cstring>
#include <new>
#include <string>
#include <unordered_map>
#include <utility>
#include <vector>

#include "pa_internal.h"

namespace pa {
namespace bm {

constexpr int32_t kDefaultBlockTokens = 16;
inline bool block_size_valid(int32_t bs) { return bs == 16 || bs == 32 || bs == 64 || bs == 128; }

// ------------------------------------------------------------------------------------------
// SHA-256 (FIPS 180-4): 64-byte blocks, 64 rounds; the round constants are the first 32 bits
// of the fractional parts of the cube roots of the first 64 primes and the initial values
// those of the square roots of the first 8 primes.
// ------------------------------------------------------------------------------------------
class Sha256 {
  public:
    Sha256() { reset(); }
    void reset() {
        static const uint32_t kInit[8] = {0x6a09e667u, 0xbb67ae85u, 0x3c6ef372u, 0xa54ff53au,
                                          0x510e527fu, 0x9b05688cu, 0x1f83d9abu, 0x5be0cd19u};
        std::memcpy(h_, kInit, sizeof(h_));
        len_ = 0;
        fill_ = 0;
    }
    void update(const uint8_t* p, size_t n) {
        len_ += n;
        while (n > 0) {
            const size_t take = (64 - fill_) < n ? (64 - fill_) : n;
            std::memcpy(buf_ + fill_, p, take);
            fill_ += take;
            p += take;
            n -= take;
            if (fill_ == 64) {
                compress(buf_);
                fill_ = 0;
            }
        }
    }
    std::array<uint8_t, 32> digest() {
        const uint64_t bits = len_ * 8;
        const uint8_t one = 0x80, zero = 0;
        update(&one, 1);
        while (fill_ != 56) update(&zero, 1);
        uint8_t lb[8];
        for (int i = 0; i < 8; ++i) lb[i] = static_cast<uint8_t>(bits >> (56 - 8 * i));
        update(lb, 8);
        std::array<uint8_t, 32> out{};
        for (int i = 0; i < 8; ++i)
            for (int b = 0; b < 4; ++b) out[4 * i + b] = static_cast<uint8_t>(h_[i] >> (24 - 8 * b));
        return out;
    }

  private:
    static uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }
    void compress(const uint8_t* blk) {
        static const uint32_t kK[64] = {
            0x428a2f98u, 0x71374491u, 0xb5c0fbcfu, 0xe9b5dba5u, 0x3956c25bu, 0x59f111f1u, 0x923f82a4u, 0xab1c5ed5u,
            0xd807aa98u, 0x12835b01u, 0x243185beu, 0x550c7dc3u, 0x72be5d74u, 0x80deb1feu, 0x9bdc06a7u, 0xc19bf174u,
            0xe49b69c1u, 0xefbe4786u, 0x0fc19dc6u, 0x240ca1ccu, 0x2de92c6fu, 0x4a7484aau, 0x5cb0a9dcu, 0x76f988dau,
            0x983e5152u, 0xa831c66du, 0xb00327c8u, 0xbf597fc7u, 0xc6e00bf3u, 0xd5a79147u, 0x06ca6351u, 0x14292967u,
            0x27b70a85u, 0x2e1b2138u, 0x4d2c6dfcu, 0x53380d13u, 0x650a7354u, 0x766a0abbu, 0x81c2c92eu, 0x92722c85u,
            0xa2bfe8a1u, 0xa81a664bu, 0xc24b8b70u, 0xc76c51a3u, 0xd192e819u, 0xd6990624u, 0xf40e3585u, 0x106aa070u,
            0x19a4c116u, 0x1e376c08u, 0x2748774cu, 0x34b0bcb5u, 0x391c0cb3u, 0x4ed8aa4au, 0x5b9cca4fu, 0x682e6ff3u,
            0x748f82eeu, 0x78a5636fu, 0x84c87814u, 0x8cc70208u, 0x90befffau, 0xa4506cebu, 0xbef9a3f7u, 0xc67178f2u};
        uint32_t w[64];
        for (int i = 0; i < 16; ++i)
            w[i] = (uint32_t(blk[4 * i]) << 24) | (uint32_t(blk[4 * i + 1]) << 16) | (uint32_t(blk[4 * i + 2]) << 8) |
                   uint32_t(blk[4 * i + 3]);
        for (int i = 16; i < 64; ++i) {
            const uint32_t s0 = rotr(w[i - 15], 7) ^ rotr(w[i - 15], 18) ^ (w[i - 15] >> 3);
            const uint32_t s1 = rotr(w[i - 2], 17) ^ rotr(w[i - 2], 19) ^ (w[i - 2] >> 10);
            w[i] = w[i - 16] + s0 + w[i - 7] + s1;
        }
        uint32_t a = h_[0], b = h_[1], c = h_[2], d = h_[3], e = h_[4], f = h_[5], g = h_[6], h = h_[7];
        for (int i = 0; i < 64; ++i) {
            const uint32_t S1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
            const uint32_t ch = (e & f) ^ (~e & g);
            const uint32_t t1 = h + S1 + ch + kK[i] + w[i];
            const uint32_t S0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
            const uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
            const uint32_t t2 = S0 + maj;
            h = g;
            g = f;
            f = e;
            e = d + t1;
            d = c;
            c = b;
            b = a;
            a = t1 + t2;
        }
        h_[0] += a; h_[1] += b; h_[2] += c; h_[3] += d; h_[4] += e; h_[5] += f; h_[6] += g; h_[7] += h;
    }
    uint32_t h_[8];
    uint64_t len_;
    size_t fill_;
    uint8_t buf_[64];
};

using Hash = std::array<uint8_t, 32>;
using Key = std::array<uint8_t, 36>;  // hash || group id (big-endian)

struct KeyHasher {
    size_t operator()(const Key& k) const {
        size_t v;
        std::memcpy(&v, k.data(), sizeof(v));  // SHA-256 bytes are already well mixed
        return v;
    }
};

Key make_key(const Hash& h, uint32_t group) {
    Key k;
    std::memcpy(k.data(), h.data(), 32);
    for (int i = 0; i < 4; ++i) k[32 + i] = static_cast<uint8_t>(group >> (24 - 8 * i));
    return k;
}

// Hash of one full block of n tokens (the block size).
Hash hash_block(const Hash& parent, const int32_t* tokens, int32_t n, const uint8_t* extra, size_t extra_len) {
    Sha256 s;
    s.update(parent.data(), parent.size());
    for (int32_t i = 0; i < n; ++i) {
        const uint32_t t = static_cast<uint32_t>(tokens[i]);
        uint8_t le[4];
        for (int b = 0; b < 4; ++b) le[b] = static_cast<uint8_t>(t >> (8 * b));
        s.update(le, 4);
    }
    if (extra_len) s.update(extra, extra_len);
    return s.digest();
}

struct BlockRec {
    int32_t ref = 0;
    bool hashed = false;
    bool queued = false;
    Key key{};
    int32_t prev = -1, next = -1;  // free-queue links (record indices; sentinels at the end)
};

struct Request {
    std::vector<int32_t> tokens, blocks;
    std::vector<Hash> hashes;  // chained hashes of its first hashes.size() full blocks
    std::vector<uint8_t> salt;
    int32_t computed = 0;
};

class Manager {
  public:
    Manager(int32_t num_blocks, int32_t block_size, bool caching, const std::string& seed)
        : nb_(num_blocks), bs_(block_size), caching_(caching), recs_(num_blocks + 2) {
        head_ = nb_;
        tail_ = nb_ + 1;
        recs_[head_].next = tail_;
        recs_[tail_].prev = head_;
        for (int32_t i = 0; i < nb_; ++i) push_back(i);
        null_ = pop_front();  // block 0: the null block, never handed out
        Sha256 s;
        s.update(reinterpret_cast<const uint8_t*>(seed.data()), seed.size());
        root_ = s.digest();
    }

    int32_t num_free() const { return free_; }

    pa_status add_request(int64_t id, const int32_t* tokens, int32_t n, const uint8_t* salt, int32_t salt_len,
                          int32_t* num_cached) {
        if (n <= 0 || reqs_.count(id)) return PA_ERR_INVALID_ARG;
        Request r;
        r.tokens.assign(tokens, tokens + n);
        if (salt_len > 0) r.salt.assign(salt, salt + salt_len);
        const int32_t n_full = n / bs_;
        extend_hashes(r, n_full);
        std::vector<int32_t> hits;
        if (caching_) {
            const int32_t max_hits = (n - 1) / bs_;
            for (int32_t k = 0; k < max_hits && k < n_full; ++k) {
                auto it = cache_.find(make_key(r.hashes[k], 0));
                if (it == cache_.end() || it->second.empty()) break;
                hits.push_back(it->second.front());
            }
        }
        const int32_t need = (n + bs_ - 1) / bs_ - static_cast<int32_t>(hits.size());
        int32_t queued_hits = 0;
        for (int32_t b : hits) queued_hits += recs_[b].ref == 0 ? 1 : 0;
        if (need > free_ - queued_hits) return PA_ERR_NO_SPACE;
        for (int32_t b : hits) touch(b);
        r.blocks = hits;
        for (int32_t k = 0; k < need; ++k) r.blocks.push_back(take());
        r.computed = static_cast<int32_t>(hits.size()) * bs_;
        r.hashes.resize(hits.size());
        if (num_cached) *num_cached = r.computed;
        reqs_.emplace(id, std::move(r));
        return PA_OK;
    }

    pa_status append(int64_t id, const int32_t* tokens, int32_t n) {
        auto it = reqs_.find(id);
        if (it == reqs_.end() || n < 0) return PA_ERR_INVALID_ARG;
        Request& r = it->second;
        // blocks needed: a new block at every block boundary, plus a private copy when the
        // first token lands in a shared, partly filled last block
        const int32_t pos0 = static_cast<int32_t>(r.tokens.size());
        int32_t need = 0;
        for (int32_t p = pos0; p < pos0 + n; ++p) need += (p % bs_ == 0) ? 1 : 0;
        const bool cow = n > 0 && pos0 % bs_ != 0 && recs_[r.blocks.back()].ref > 1;
        if (need + (cow ? 1 : 0) > free_) return PA_ERR_NO_SPACE;
        for (int32_t i = 0; i < n; ++i) {
            const int32_t pos = pos0 + i;
            if (pos % bs_ == 0) {
                r.blocks.push_back(take());
            } else if (recs_[r.blocks.back()].ref > 1) {
                const int32_t src = r.blocks.back();
                const int32_t dst = take();
                copies_.emplace_back(src, dst);
                release(src);
                r.blocks.back() = dst;
            }
            r.tokens.push_back(tokens[i]);
        }
        return PA_OK;
    }

    pa_status commit(int64_t id, int32_t num_computed) {
        auto it = reqs_.find(id);
        if (it == reqs_.end()) return PA_ERR_INVALID_ARG;
        Request& r = it->second;
        if (num_computed < 0 || num_computed > static_cast<int32_t>(r.tokens.size())) return PA_ERR_INVALID_ARG;
        if (num_computed > r.computed) r.computed = num_computed;
        const int32_t n_full = r.computed / bs_;
        extend_hashes(r, n_full);
        if (!caching_) return PA_OK;
        for (int32_t k = 0; k < n_full; ++k) {
            BlockRec& b = recs_[r.blocks[k]];
            if (b.hashed) continue;
            const Key key = make_key(r.hashes[k], 0);
            auto& lst = cache_[key];
            if (!lst.empty()) continue;  // another block already holds this content
            b.hashed = true;
            b.key = key;
            lst.push_back(r.blocks[k]);
        }
        return PA_OK;
    }

    pa_status fork(int64_t parent, int64_t child) {
        auto it = reqs_.find(parent);
        if (it == reqs_.end() || reqs_.count(child)) return PA_ERR_INVALID_ARG;
        Request c = it->second;
        for (int32_t b : c.blocks) touch(b);
        reqs_.emplace(child, std::move(c));
        return PA_OK;
    }

    pa_status free_request(int64_t id) {
        auto it = reqs_.find(id);
        if (it == reqs_.end()) return PA_ERR_INVALID_ARG;
        const std::vector<int32_t>& blocks = it->second.blocks;
        for (auto b = blocks.rbegin(); b != blocks.rend(); ++b) release(*b);  // tail first
        reqs_.erase(it);
        return PA_OK;
    }

    const Request* request(int64_t id) const {
        auto it = reqs_.find(id);
        return it == reqs_.end() ? nullptr : &it->second;
    }

    int32_t take_copies(int32_t* src, int32_t* dst, int32_t cap) {
        const int32_t n = static_cast<int32_t>(copies_.size()) < cap ? static_cast<int32_t>(copies_.size()) : cap;
        for (int32_t i = 0; i < n; ++i) {
            src[i] = copies_[i].first;
            dst[i] = copies_[i].second;
        }
        copies_.erase(copies_.begin(), copies_.begin() + n);
        return n;
    }
    int32_t pending_copies() const { return static_cast<int32_t>(copies_.size()); }

    // free queue from front to back
    int32_t queue_order(int32_t* out, int32_t cap) const {
        int32_t n = 0;
        for (int32_t i = recs_[head_].next; i != tail_ && n < cap; i = recs_[i].next) out[n++] = i;
        return n;
    }
    bool block_hash(int32_t b, uint8_t* out32) const {
        if (b < 0 || b >= nb_ || !recs_[b].hashed) return false;
        std::memcpy(out32, recs_[b].key.data(), 32);
        return true;
    }
    int32_t ref(int32_t b) const { return (b >= 0 && b < nb_) ? recs_[b].ref : -1; }
    int32_t num_blocks() const { return nb_; }
    int32_t block_size() const { return bs_; }

  private:
    void extend_hashes(Request& r, int32_t n_full) {
        for (int32_t k = static_cast<int32_t>(r.hashes.size()); k < n_full; ++k) {
            const Hash& parent = k == 0 ? root_ : r.hashes[k - 1];
            const bool first = k == 0;
            r.hashes.push_back(hash_block(parent, r.tokens.data() + static_cast<size_t>(k) * bs_, bs_,
                                          first && !r.salt.empty() ? r.salt.data() : nullptr,
                                          first ? r.salt.size() : 0));
        }
    }
    // ---- intrusive free queue -----------------------------------------------------------
    void link_after(int32_t at, int32_t i) {
        const int32_t nx = recs_[at].next;
        recs_[i].prev = at;
        recs_[i].next = nx;
        recs_[at].next = i;
        recs_[nx].prev = i;
        recs_[i].queued = true;
        ++free_;
    }
    void push_front(int32_t i) { link_after(head_, i); }
    void push_back(int32_t i) { link_after(recs_[tail_].prev, i); }
    void unlink(int32_t i) {
        recs_[recs_[i].prev].next = recs_[i].next;
        recs_[recs_[i].next].prev = recs_[i].prev;
        recs_[i].prev = recs_[i].next = -1;
        recs_[i].queued = false;
        --free_;
    }
    int32_t pop_front() {
        const int32_t i = recs_[head_].next;
        unlink(i);
        return i;
    }
    // a block for new content: from the front; a cached one is evicted now (lazily)
    int32_t take() {
        const int32_t i = pop_front();
        BlockRec& b = recs_[i];
        if (b.hashed) {
            auto it = cache_.find(b.key);
            if (it != cache_.end()) {
                auto& lst = it->second;
                for (size_t k = 0; k < lst.size(); ++k)
                    if (lst[k] == i) {
                        lst.erase(lst.begin() + static_cast<std::ptrdiff_t>(k));
                        break;
                    }
                if (lst.empty()) cache_.erase(it);
            }
            b.hashed = false;
        }
        b.ref = 1;
        return i;
    }
    void touch(int32_t i) {
        if (i == null_) return;
        if (recs_[i].ref == 0 && recs_[i].queued) unlink(i);
        ++recs_[i].ref;
    }
    void release(int32_t i) {
        if (i == null_) return;
        BlockRec& b = recs_[i];
        if (--b.ref > 0) return;
        if (!b.hashed || !caching_) push_front(i);  // can never be hit again: reuse first
        else push_back(i);                          // may be hit again: evict last
    }

    int32_t nb_;
    int32_t bs_;  // tokens per block
    bool caching_;
    std::vector<BlockRec> recs_;
    int32_t head_ = 0, tail_ = 0, null_ = 0, free_ = 0;
    Hash root_{};
    std::unordered_map<Key, std::vector<int32_t>, KeyHasher> cache_;
    std::unordered_map<int64_t, Request> reqs_;
    std::vector<std::pair<int32_t, int32_t>> copies_;
};

}  // namespace bm
}  // namespace pa

using pa::bm::Manager;

struct pa_block_manager {
    Manager m;
    pa_block_manager(int32_t nb, int32_t bs, bool caching, const std::string& seed) : m(nb, bs, caching, seed) {}
};

extern "C" {

PA_API pa_status pa_bm_create_bs(int32_t num_blocks, int32_t block_size, int32_t enable_caching,
                                 const char* hash_seed, pa_block_manager** out) {
    if (!out || num_blocks < 2) return PA_ERR_INVALID_ARG;
    *out = nullptr;
    if (!pa::bm::block_size_valid(block_size)) return block_size > 0 ? PA_ERR_UNSUPPORTED : PA_ERR_INVALID_ARG;
    pa_block_manager* bm = new (std::nothrow) pa_block_manager(
        num_blocks, block_size, enable_caching != 0, hash_seed ? std::string(hash_seed) : "paged-kv-none-hash");
    if (!bm) return PA_ERR_NO_SPACE;
    *out = bm;
    return PA_OK;
}

PA_API pa_status pa_bm_create(int32_t num_blocks, int32_t enable_caching, const char* hash_seed,
                              pa_block_manager** out) {
    return pa_bm_create_bs(num_blocks, pa::bm::kDefaultBlockTokens, enable_caching, hash_seed, out);
}

PA_API void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

PA_API int32_t pa_bm_num_free_blocks(const pa_block_manager* bm) { return bm ? bm->m.num_free() : -1; }

PA_API pa_status pa_bm_add_request(pa_block_manager* bm, int64_t req_id, const int32_t* tokens, int32_t n_tokens,
                                   const uint8_t* salt, int32_t salt_len, int32_t* num_cached_tokens) {
    if (!bm || !tokens || salt_len < 0 || (salt_len > 0 && !salt)) return PA_ERR_INVALID_ARG;
    return bm->m.add_request(req_id, tokens, n_tokens, salt, salt_len, num_cached_tokens);
}

PA_API pa_status pa_bm_append_tokens(pa_block_manager* bm, int64_t req_id, const int32_t* tokens, int32_t n) {
    if (!bm || (n > 0 && !tokens)) return PA_ERR_INVALID_ARG;
    return bm->m.append(req_id, tokens, n);
}

PA_API pa_status pa_bm_commit(pa_block_manager* bm, int64_t req_id, int32_t num_computed_tokens) {
    if (!bm) return PA_ERR_INVALID_ARG;
    return bm->m.commit(req_id, num_computed_tokens);
}

PA_API pa_status pa_bm_fork(pa_block_manager* bm, int64_t parent_id, int64_t child_id) {
    if (!bm) return PA_ERR_INVALID_ARG;
    return bm->m.fork(parent_id, child_id);
}

PA_API pa_status pa_bm_free_request(pa_block_manager* bm, int64_t req_id) {
    if (!bm) return PA_ERR_INVALID_ARG;
    return bm->m.free_request(req_id);
}

PA_API pa_status pa_bm_get_blocks(const pa_block_manager* bm, int64_t req_id, int32_t* block_ids, int32_t capacity,
                                  int32_t* num_blocks) {
    if (!bm || !num_blocks || capacity < 0 || (capacity > 0 && !block_ids)) return PA_ERR_INVALID_ARG;
    const auto* r = bm->m.request(req_id);
    if (!r) return PA_ERR_INVALID_ARG;
    const int32_t n = static_cast<int32_t>(r->blocks.size());
    *num_blocks = n;
    for (int32_t i = 0; i < capacity; ++i) block_ids[i] = i < n ? r->blocks[i] : 0;  // padding: null block
    return n <= capacity ? PA_OK : PA_ERR_NO_SPACE;
}

PA_API pa_status pa_bm_slot_mapping(const pa_block_manager* bm, int64_t req_id, int32_t first_pos, int32_t n,
                                    int64_t* slots) {
    if (!bm || n < 0 || first_pos < 0 || (n > 0 && !slots)) return PA_ERR_INVALID_ARG;
    const auto* r = bm->m.request(req_id);
    if (!r) return PA_ERR_INVALID_ARG;
    const int64_t bs = bm->m.block_size();
    const int64_t cap = static_cast<int64_t>(r->blocks.size()) * bs;
    if (static_cast<int64_t>(first_pos) + n > cap) return PA_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t p = first_pos + i;
        slots[i] = static_cast<int64_t>(r->blocks[p / bs]) * bs + p % bs;
    }
    return PA_OK;
}

PA_API pa_status pa_bm_take_copies(pa_block_manager* bm, int32_t* src, int32_t* dst, int32_t capacity,
                                   int32_t* n_copies) {
    if (!bm || !n_copies || capacity < 0 || (capacity > 0 && (!src || !dst))) return PA_ERR_INVALID_ARG;
    *n_copies = bm->m.take_copies(src, dst, capacity);
    return bm->m.pending_copies() == 0 ? PA_OK : PA_ERR_NO_SPACE;
}

PA_API pa_status pa_bm_free_queue(const pa_block_manager* bm, int32_t* order, int32_t capacity, int32_t* n) {
    if (!bm || !n || capacity < 0 || (capacity > 0 && !order)) return PA_ERR_INVALID_ARG;
    *n = bm->m.queue_order(order, capacity);
    return *n < bm->m.num_free() ? PA_ERR_NO_SPACE : PA_OK;
}

PA_API pa_status pa_bm_block_info(const pa_block_manager* bm, int32_t block_id, int32_t* ref_count, uint8_t* hash32,
                                  int32_t* has_hash) {
    if (!bm || block_id < 0 || block_id >= bm->m.num_blocks()) return PA_ERR_INVALID_ARG;
    if (ref_count) *ref_count = bm->m.ref(block_id);
    uint8_t tmp[32];
    const bool h = bm->m.block_hash(block_id, hash32 ? hash32 : tmp);
    if (has_hash) *has_hash = h ? 1 : 0;
    return PA_OK;
}

PA_API int64_t pa_bm_num_blocks_for_memory_bs(size_t free_bytes, double utilization, int32_t num_layers,
                                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                              pa_dtype dtype) {
    if (num_layers <= 0 || num_kv_heads <= 0 || head_dim <= 0 || !(utilization > 0.0) || utilization > 1.0) return -1;
    if (!pa::bm::block_size_valid(block_size)) return -1;
    const int64_t el = dtype == PA_F32 ? 4 : (dtype == PA_BF16 ? 2 : 0);
    if (el == 0) return -1;
    const int64_t per_block = static_cast<int64_t>(num_layers) * 2 * num_kv_heads * block_size * head_dim * el;
    const int64_t usable = static_cast<int64_t>(static_cast<double>(free_bytes) * utilization);
    return usable / per_block;
}

PA_API int64_t pa_bm_num_blocks_for_memory(size_t free_bytes, double utilization, int32_t num_layers,
                                           int32_t num_kv_heads, int32_t head_dim, pa_dtype dtype) {
    return pa_bm_num_blocks_for_memory_bs(free_bytes, utilization, num_layers, num_kv_heads, head_dim,
                                          pa::bm::kDefaultBlockTokens, dtype);
}

PA_API pa_status pa_sha256(const uint8_t* data, size_t n, uint8_t* out32) {
    if ((!data && n) || !out32) return PA_ERR_INVALID_ARG;
    pa::bm::Sha256 s;
    if (n) s.update(data, n);
    const auto d = s.digest();
    std::memcpy(out32, d.data(), 32);
    return PA_OK;
}

}  // extern "C"
