// block_manager.cpp -- host allocator of the paged KV pool (declared in pagedkv.h).
//
// What it models ("注意力演进与推理流程", 变革 1 and 变革 3; xinc.fun archive 233,
// section 6): the cache is cut into fixed-size blocks of 16 tokens, a sequence
// gets a new block whenever it crosses a block boundary, sequences that share a
// prefix (or parallel candidates forked from one sequence) reference the same
// physical blocks until they branch, and a prompt whose leading blocks were
// computed before can take those blocks over instead of recomputing them.
//
// Invariants kept by every call (checked by the CPU tests after every step):
//  * ref[b] = number of sequences whose table contains b (with multiplicity);
//  * b is in exactly one of {held (ref > 0), plain free list, published free list};
//  * no slot handed out by an append lies in a block with ref > 1;
//  * a call that returns an error leaves the manager unchanged: every host
//    allocation a call needs happens before its first change, and a failed one
//    (std::bad_alloc, caught at the C boundary) is reported as
//    PKV_ERR_OUT_OF_BLOCKS.
#include <algorithm>
#include <array>
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

namespace {

constexpr int32_t kBlock = 16;  // tokens per block

// One published full block: the hash of all token ids up to its end, and (to
// rule out collisions) its own 16 ids and the hash of the prefix before it.
struct Published {
    uint64_t hash = 0;
    uint64_t parent = 0;
    std::array<int32_t, kBlock> tokens{};
};

struct BlockInfo {
    int32_t ref = 0;
    bool published = false;
    Published pub;
    bool in_lru = false;  // free and published: linked into the LRU list below
    int32_t prev = -1, next = -1;
};

struct Seq {
    std::vector<int32_t> blocks;
    int64_t len = 0;
};

// Hash of a block's ids chained onto the prefix hash (splitmix64 finaliser per word).
uint64_t mix(uint64_t x) {
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

uint64_t chain_hash(uint64_t parent, const int32_t *tokens) {
    uint64_t h = mix(parent ^ 0x5851F42D4C957F2Dull);
    for (int i = 0; i < kBlock; ++i) h = mix(h ^ static_cast<uint32_t>(tokens[i]));
    return h;
}

// Runs f, mapping a host allocation failure to an error code (no exception crosses the C ABI).
template <class F>
int guarded(F &&f) {
    try {
        return f();
    } catch (...) {
        return PKV_ERR_OUT_OF_BLOCKS;
    }
}

}  // namespace

struct pkv_block_manager {
    std::vector<BlockInfo> info;
    std::vector<int32_t> plain_free;  // unpublished free blocks (stack; capacity num_blocks)
    // Published free blocks, oldest first: an intrusive list through info[].prev/next,
    // so releasing a block never allocates.
    int32_t lru_head = -1, lru_tail = -1, lru_size = 0;
    std::unordered_map<uint64_t, int32_t> by_hash;
    std::unordered_map<int64_t, Seq> seqs;

    int32_t num_free() const { return static_cast<int32_t>(plain_free.size()) + lru_size; }

    void lru_push_back(int32_t b) {
        BlockInfo &bi = info[b];
        bi.prev = lru_tail;
        bi.next = -1;
        if (lru_tail >= 0) info[lru_tail].next = b; else lru_head = b;
        lru_tail = b;
        bi.in_lru = true;
        ++lru_size;
    }

    void lru_remove(int32_t b) {
        BlockInfo &bi = info[b];
        if (bi.prev >= 0) info[bi.prev].next = bi.next; else lru_head = bi.next;
        if (bi.next >= 0) info[bi.next].prev = bi.prev; else lru_tail = bi.prev;
        bi.prev = bi.next = -1;
        bi.in_lru = false;
        --lru_size;
    }

    void unpublish(int32_t b) {
        BlockInfo &bi = info[b];
        if (!bi.published) return;
        auto it = by_hash.find(bi.pub.hash);
        if (it != by_hash.end() && it->second == b) by_hash.erase(it);
        bi.published = false;
    }

    // Caller has checked num_free() > 0.
    int32_t allocate() {
        int32_t b;
        if (!plain_free.empty()) {
            b = plain_free.back();
            plain_free.pop_back();
        } else {
            b = lru_head;  // the oldest published free block
            lru_remove(b);
            unpublish(b);  // its contents are about to be overwritten
        }
        info[b].ref = 1;
        return b;
    }

    void retain(int32_t b) {
        BlockInfo &bi = info[b];
        if (bi.ref == 0 && bi.in_lru) lru_remove(b);
        ++bi.ref;
    }

    void release(int32_t b) {
        BlockInfo &bi = info[b];
        if (--bi.ref > 0) return;
        if (bi.published)
            lru_push_back(b);
        else
            plain_free.push_back(b);  // within the reserved capacity
    }
};

extern "C" {

int pkv_bm_create(int32_t num_blocks, pkv_block_manager **out) {
    if (!out || num_blocks < 1) return PKV_ERR_INVALID_ARG;
    *out = nullptr;
    pkv_block_manager *bm = new (std::nothrow) pkv_block_manager();
    if (!bm) return PKV_ERR_OUT_OF_BLOCKS;
    try {
        bm->info.resize(num_blocks);
        bm->plain_free.reserve(num_blocks);
        // Hand out low block ids first (a stack popped from the back).
        for (int32_t b = num_blocks - 1; b >= 0; --b) bm->plain_free.push_back(b);
    } catch (...) {
        delete bm;
        return PKV_ERR_OUT_OF_BLOCKS;
    }
    *out = bm;
    return PKV_OK;
}

void pkv_bm_destroy(pkv_block_manager *bm) { delete bm; }

int32_t pkv_bm_num_free(const pkv_block_manager *bm) { return bm ? bm->num_free() : 0; }

int pkv_bm_ref_count(const pkv_block_manager *bm, int32_t block, int32_t *count) {
    if (!bm || !count || block < 0 || block >= static_cast<int32_t>(bm->info.size())) return PKV_ERR_INVALID_ARG;
    *count = bm->info[block].ref;
    return PKV_OK;
}

int pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq_id) {
    if (!bm || bm->seqs.count(seq_id)) return PKV_ERR_INVALID_ARG;
    return guarded([&] {
        bm->seqs.emplace(seq_id, Seq{});
        return PKV_OK;
    });
}

int pkv_bm_fork(pkv_block_manager *bm, int64_t parent_id, int64_t child_id) {
    if (!bm || parent_id == child_id || bm->seqs.count(child_id)) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(parent_id);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
    const Seq *parent = &it->second;  // element references survive a rehash
    return guarded([&] {
        Seq child = *parent;
        bm->seqs.emplace(child_id, std::move(child));  // may throw: nothing changed yet
        for (int32_t b : parent->blocks) bm->retain(b);
        return PKV_OK;
    });
}

int pkv_bm_append(pkv_block_manager *bm, int64_t seq_id, int32_t num_tokens, int32_t *slot_mapping,
                  int32_t *copy_pair, int32_t *num_copies) {
    if (!bm || num_tokens < 0 || !num_copies || (num_tokens > 0 && (!slot_mapping || !copy_pair)))
        return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
    Seq &s = it->second;
    *num_copies = 0;
    if (num_tokens == 0) return PKV_OK;
    const int64_t new_len = s.len + num_tokens;
    if ((new_len + kBlock - 1) / kBlock > INT32_MAX) return PKV_ERR_INVALID_ARG;
    const int64_t extra = (new_len + kBlock - 1) / kBlock - static_cast<int64_t>(s.blocks.size());
    // The next token lands in the current last block only if it is partly filled.
    const bool cow = (s.len % kBlock) != 0 && bm->info[s.blocks.back()].ref > 1;
    if (extra + (cow ? 1 : 0) > bm->num_free()) return PKV_ERR_OUT_OF_BLOCKS;
    if (guarded([&] {
            s.blocks.reserve(s.blocks.size() + extra);  // the only allocation, before any change
            return PKV_OK;
        }) != PKV_OK)
        return PKV_ERR_OUT_OF_BLOCKS;
    if (cow) {
        const int32_t old = s.blocks.back();
        const int32_t fresh = bm->allocate();
        bm->release(old);
        s.blocks.back() = fresh;
        copy_pair[0] = old;
        copy_pair[1] = fresh;
        *num_copies = 1;
    }
    for (int64_t i = 0; i < extra; ++i) s.blocks.push_back(bm->allocate());
    for (int32_t t = 0; t < num_tokens; ++t) {
        const int64_t p = s.len + t;
        slot_mapping[t] = s.blocks[p / kBlock] * kBlock + static_cast<int32_t>(p % kBlock);
    }
    s.len = new_len;
    return PKV_OK;
}

int pkv_bm_append_batch(pkv_block_manager *bm, const int64_t *seq_ids, int32_t num_seqs, const int32_t *num_tokens,
                        int32_t *slot_mapping, int32_t *copy_pairs, int32_t *num_copies) {
    if (!bm || num_seqs < 0 || !num_copies || (num_seqs > 0 && (!seq_ids || !slot_mapping || !copy_pairs)))
        return PKV_ERR_INVALID_ARG;
    *num_copies = 0;
    return guarded([&] {
        // Dry run in call order: the blocks needed, with each copy-on-write decision made
        // as the real appends will make it (an earlier copy can leave a block unshared).
        std::vector<Seq *> seqs(num_seqs);
        std::unordered_map<int32_t, int32_t> dropped;  // references released earlier in this call
        std::unordered_map<int64_t, int> seen;
        int64_t need = 0;
        for (int32_t i = 0; i < num_seqs; ++i) {
            auto it = bm->seqs.find(seq_ids[i]);
            if (it == bm->seqs.end() || seen[seq_ids[i]]++) return PKV_ERR_INVALID_ARG;  // unknown or repeated
            const int32_t n = num_tokens ? num_tokens[i] : 1;
            if (n < 0) return PKV_ERR_INVALID_ARG;
            Seq &sq = it->second;
            seqs[i] = &sq;
            if (n == 0) continue;
            const int64_t new_len = sq.len + n;
            if ((new_len + kBlock - 1) / kBlock > INT32_MAX) return PKV_ERR_INVALID_ARG;
            need += (new_len + kBlock - 1) / kBlock - static_cast<int64_t>(sq.blocks.size());
            if (sq.len % kBlock != 0) {
                const int32_t last = sq.blocks.back();
                int32_t &d = dropped[last];
                if (bm->info[last].ref - d > 1) {
                    ++need;
                    ++d;
                }
            }
        }
        if (need > bm->num_free()) return PKV_ERR_OUT_OF_BLOCKS;
        for (int32_t i = 0; i < num_seqs; ++i) {  // reserve before the first change
            const int32_t n = num_tokens ? num_tokens[i] : 1;
            seqs[i]->blocks.reserve((seqs[i]->len + n + kBlock - 1) / kBlock);
        }
        int64_t off = 0;
        int32_t copies = 0;
        for (int32_t i = 0; i < num_seqs; ++i) {
            const int32_t n = num_tokens ? num_tokens[i] : 1;
            int32_t nc = 0;
            pkv_bm_append(bm, seq_ids[i], n, slot_mapping + off, copy_pairs + 2 * copies, &nc);  // cannot fail now
            off += n;
            copies += nc;
        }
        *num_copies = copies;
        return PKV_OK;
    });
}

int pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq_id) {
    if (!bm) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
    // Release from the end so a sequence's early (most shareable) blocks are freed last.
    for (auto b = it->second.blocks.rbegin(); b != it->second.blocks.rend(); ++b) bm->release(*b);
    bm->seqs.erase(it);
    return PKV_OK;
}

int pkv_bm_sequence_length(const pkv_block_manager *bm, int64_t seq_id, int64_t *length) {
    if (!bm || !length) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
    *length = it->second.len;
    return PKV_OK;
}

int pkv_bm_block_tables(const pkv_block_manager *bm, const int64_t *seq_ids, int32_t num_seqs,
                        int32_t max_blocks_per_seq, int32_t pad_block, int32_t *block_tables,
                        int32_t *context_lens) {
    if (!bm || num_seqs < 0 || max_blocks_per_seq < 1) return PKV_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!seq_ids || !block_tables || !context_lens)) return PKV_ERR_INVALID_ARG;
    // Validate every row before writing any.
    for (int32_t i = 0; i < num_seqs; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return PKV_ERR_INVALID_ARG;
        if (it->second.blocks.size() > static_cast<size_t>(max_blocks_per_seq) || it->second.len > INT32_MAX)
            return PKV_ERR_INVALID_ARG;
    }
    for (int32_t i = 0; i < num_seqs; ++i) {
        const Seq &sq = bm->seqs.find(seq_ids[i])->second;
        int32_t *row = block_tables + static_cast<int64_t>(i) * max_blocks_per_seq;
        std::copy(sq.blocks.begin(), sq.blocks.end(), row);
        std::fill(row + sq.blocks.size(), row + max_blocks_per_seq, pad_block);
        context_lens[i] = static_cast<int32_t>(sq.len);
    }
    return PKV_OK;
}

int pkv_bm_publish(pkv_block_manager *bm, int64_t seq_id, const int32_t *tokens, int32_t num_tokens) {
    if (!bm || num_tokens < 0 || (num_tokens > 0 && !tokens)) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end() || num_tokens > it->second.len) return PKV_ERR_INVALID_ARG;
    const Seq &s = it->second;
    uint64_t parent = 0;
    for (int32_t i = 0; (i + 1) * kBlock <= num_tokens; ++i) {
        const int32_t *ids = tokens + static_cast<int64_t>(i) * kBlock;
        const uint64_t h = chain_hash(parent, ids);
        const int32_t b = s.blocks[i];
        if (!bm->by_hash.count(h) && !bm->info[b].published) {
            // The map insertion is the only allocation; the block is marked after it.
            if (guarded([&] {
                    bm->by_hash.emplace(h, b);
                    return PKV_OK;
                }) != PKV_OK)
                return PKV_ERR_OUT_OF_BLOCKS;  // blocks before i stay published: each is complete
            BlockInfo &bi = bm->info[b];
            bi.published = true;
            bi.pub.hash = h;
            bi.pub.parent = parent;
            std::copy(ids, ids + kBlock, bi.pub.tokens.begin());
        }
        parent = h;
    }
    return PKV_OK;
}

int pkv_bm_add_sequence_cached(pkv_block_manager *bm, int64_t seq_id, const int32_t *tokens, int32_t num_tokens,
                               int32_t *num_cached_tokens) {
    if (!bm || num_tokens < 0 || !num_cached_tokens || (num_tokens > 0 && !tokens) || bm->seqs.count(seq_id))
        return PKV_ERR_INVALID_ARG;
    return guarded([&] {
        Seq s;
        uint64_t parent = 0;
        // Leave at least one prompt token to compute: take blocks ending before num_tokens.
        for (int32_t i = 0; (i + 1) * kBlock < num_tokens; ++i) {
            const int32_t *ids = tokens + static_cast<int64_t>(i) * kBlock;
            const uint64_t h = chain_hash(parent, ids);
            auto hit = bm->by_hash.find(h);
            if (hit == bm->by_hash.end()) break;
            const Published &pub = bm->info[hit->second].pub;
            if (pub.parent != parent || !std::equal(ids, ids + kBlock, pub.tokens.begin())) break;
            s.blocks.push_back(hit->second);
            parent = h;
        }
        s.len = static_cast<int64_t>(s.blocks.size()) * kBlock;
        const int32_t cached = static_cast<int32_t>(s.len);
        const std::vector<int32_t> taken = s.blocks;
        bm->seqs.emplace(seq_id, std::move(s));  // last allocation; then the counts change
        for (int32_t b : taken) bm->retain(b);
        *num_cached_tokens = cached;
        return PKV_OK;
    });
}

}  // extern "C"
