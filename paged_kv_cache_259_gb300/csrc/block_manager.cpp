// Host block manager: free list, per-sequence block tables, reference counts,
// fork and block-level copy-on-write.
//
// "PagedAttention" (Ultralytics glossary), "Cách phân trang hoạt động": blocks of
// a fixed number of tokens, a new block only when the last one is full, taken
// from wherever a free block is (the worked example pops the front of a list of
// scattered ids), the block table recording the order.
// "KV cache paginado e batching contínuo para LLMs", "Como funciona": several
// logical blocks may map to one physical block with a reference count; writing
// into a shared block allocates another, copies, and decrements the original.
// Glossary, "Batching liên tục": a finished sequence's blocks return to the pool
// at once.
//
// Host memory only; no CUDA. The manager never touches KV data: it hands out
// slot numbers and (src, dst) copy pairs that the device calls consume.
//
// Prefix caching (optional; glossary "Chia sẻ block giữa các chuỗi": requests
// that begin with the same system prompt reuse one copy of the common prefix;
// the vLLM feature list names prefix caching): a block filled by tokens whose
// ids are known is registered under its prefix -- every token id from the start
// of the sequence to the end of the block. A new request reuses, from the front,
// the registered blocks of its prompt (leaving at least one prompt token to
// compute); a registered block whose count reaches 0 stays cached as evictable
// (revived by a later hit) until a new block is needed and the free list is
// empty, when the oldest evictable block is evicted. Within one release,
// uncached blocks go to the free list in table order and cached ones to the
// evictable list in reverse table order. The index is a 64-bit hash of the whole
// prefix (chained block by block); a hit also compares the block's own token
// ids and the hash of the prefix before it.
//
// Beam search (glossary, "Chia sẻ block giữa các chuỗi": beams share blocks with
// a count per block and copy a shared block before writing into it): one step's
// reshuffle forks every new beam from its parent, in order, then frees the old
// beams in order; the new beams' appends then copy shared partial blocks.
//
// Swapping ("KV cache paginado...", "Como funciona": when physical blocks run
// out the newest requests are preempted, all or nothing, and their blocks
// recovered by swapping to the CPU or by recomputation): a host pool of blocks
// with its own free list; swapping a sequence out gives each block of its table,
// in order, a fresh host block and a (device, host) copy pair and releases the
// device blocks as a free does; swapping in is the reverse onto fresh device
// blocks. Either is refused, changing nothing, if the receiving pool cannot take
// the whole sequence. A swapped-out sequence can only be swapped in or freed.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <deque>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pagedkv.h"

namespace {

constexpr int64_t kUnknownToken = INT64_MIN;
constexpr uint64_t kPrefixSeed = 0x243f6a8885a308d3ULL;

// splitmix64's output function (Steele, Lea, Flood: "Fast splittable
// pseudorandom number generators"), used to chain token ids into a prefix hash.
uint64_t mix64(uint64_t x) {
    x ^= x >> 30;
    x *= 0xbf58476d1ce4e5b9ULL;
    x ^= x >> 27;
    x *= 0x94d049bb133111ebULL;
    x ^= x >> 31;
    return x;
}

uint64_t chain(uint64_t h, const int64_t* tok, int n) {
    for (int i = 0; i < n; ++i) h = mix64(h ^ (mix64((uint64_t)tok[i]) + 0x9e3779b97f4a7c15ULL));
    return h;
}

}  // namespace

struct pkv_block_manager {
    int num_blocks = 0;
    int block_size = 0;
    std::deque<int32_t> free_list;       // front = next block handed out
    std::vector<int32_t> ref;            // reference count per physical block
    struct Seq {
        std::vector<int32_t> table;      // logical block i -> physical block id
        int64_t len = 0;                 // tokens cached
        std::vector<int64_t> tokens;     // token ids (prefix caching only)
        std::vector<uint64_t> hashes;    // prefix hash after each full block
        bool swapped = false;            // table holds host blocks
        uint64_t demand_epoch = 0;       // Demand scratch: length within a batch count
        int64_t demand_len = 0;
    };
    std::unordered_map<int64_t, Seq> seqs;

    // ---- prefix caching
    bool caching = false;
    std::vector<char> registered;                    // block holds a registered prefix
    std::vector<uint64_t> key_hash, parent_hash;     // hash through / before the block
    std::vector<int64_t> block_tokens;               // num_blocks x block_size ids
    std::unordered_multimap<uint64_t, int32_t> index;
    std::list<int32_t> evictable;                    // registered, count 0; oldest first
    std::vector<std::list<int32_t>::iterator> ev_pos;
    std::vector<char> in_ev;
    int64_t hit_blocks = 0, lookup_blocks = 0;

    // ---- Demand scratch: references given up by CoW within one batch count,
    // valid where drop_epoch matches the count's epoch (no clearing per batch)
    uint64_t epoch = 0;
    std::vector<uint64_t> drop_epoch;
    std::vector<int32_t> drop_count;

    // ---- host pool (swapping)
    int num_host_blocks = 0;
    std::deque<int32_t> host_free;                   // front = next host block

    size_t device_available() const {
        return free_list.size() + (caching ? evictable.size() : 0);
    }

    // Drop one reference to each device block of `table`: uncached blocks that
    // reach 0 go to the free list in table order, cached ones to the evictable
    // list in reverse table order.
    void release(const std::vector<int32_t>& table) {
        std::vector<int32_t> cached;
        for (int32_t b : table) {
            ref[b] -= 1;
            if (ref[b] == 0) {
                if (caching && registered[b])
                    cached.push_back(b);
                else
                    free_list.push_back(b);
            }
        }
        for (auto r = cached.rbegin(); r != cached.rend(); ++r) {
            ev_pos[*r] = evictable.insert(evictable.end(), *r);
            in_ev[*r] = 1;
        }
    }

    bool can_take() const { return !free_list.empty() || (caching && !evictable.empty()); }

    void deregister(int32_t b) {
        auto range = index.equal_range(key_hash[b]);
        for (auto it = range.first; it != range.second; ++it)
            if (it->second == b) {
                index.erase(it);
                break;
            }
        registered[b] = 0;
    }

    int32_t take() {
        int32_t b;
        if (!free_list.empty()) {
            b = free_list.front();
            free_list.pop_front();
        } else {                                     // caller checked can_take()
            b = evictable.front();
            evictable.pop_front();
            in_ev[b] = 0;
            deregister(b);
        }
        ref[b] = 1;
        return b;
    }

    // Registered block holding the block after prefix hash `parent` with these
    // token ids, or -1.
    int32_t find(uint64_t parent, uint64_t key, const int64_t* tok) const {
        auto range = index.equal_range(key);
        for (auto it = range.first; it != range.second; ++it) {
            const int32_t b = it->second;
            if (parent_hash[b] != parent) continue;
            bool same = true;
            for (int i = 0; i < block_size && same; ++i)
                same = block_tokens[(size_t)b * block_size + i] == tok[i];
            if (same) return b;
        }
        return -1;
    }

    // The sequence's last block has just been filled: register it under its
    // prefix unless a token id is unknown or the prefix is registered already.
    void maybe_register(Seq& s) {
        const int64_t nb = s.len / block_size;
        // the chain stops at the first block with an unknown token id
        if (s.hashes.size() != (size_t)(nb - 1)) return;
        const int64_t* tok = s.tokens.data() + (nb - 1) * block_size;
        for (int i = 0; i < block_size; ++i)
            if (tok[i] == kUnknownToken) return;
        const uint64_t parent = nb > 1 ? s.hashes[nb - 2] : kPrefixSeed;
        const uint64_t key = chain(parent, tok, block_size);
        s.hashes.push_back(key);
        const int32_t b = s.table.back();
        if (registered[b] || find(parent, key, tok) >= 0) return;
        registered[b] = 1;
        key_hash[b] = key;
        parent_hash[b] = parent;
        for (int i = 0; i < block_size; ++i) block_tokens[(size_t)b * block_size + i] = tok[i];
        index.emplace(key, b);
    }

    // One append; on exhaustion nothing changes.
    int append(Seq& s, int64_t token, int64_t* slot, int32_t* cow_src, int32_t* cow_dst) {
        *cow_src = -1;
        *cow_dst = -1;
        if (s.swapped) return PKV_ERR_INVALID_ARG;
        const int64_t n = s.len;
        if (n % block_size == 0) {
            if (!can_take()) return PKV_ERR_POOL_EXHAUSTED;
            s.table.push_back(take());
        } else {
            const int32_t last = s.table.back();
            if (ref[last] > 1) {                       // shared: copy before writing
                if (!can_take()) return PKV_ERR_POOL_EXHAUSTED;
                const int32_t dst = take();
                ref[last] -= 1;
                s.table.back() = dst;
                *cow_src = last;
                *cow_dst = dst;
            }
        }
        const int32_t block = s.table[n / block_size];
        *slot = (int64_t)block * block_size + n % block_size;
        s.len = n + 1;
        if (caching) {
            s.tokens.push_back(token);
            if (s.len % block_size == 0) maybe_register(s);
        }
        return PKV_OK;
    }

    int append(Seq& s, int64_t* slot, int32_t* cow_src, int32_t* cow_dst) {
        return append(s, kUnknownToken, slot, cow_src, cow_dst);
    }

    // What a batch of appends would take, found without changing anything, so
    // that a batch either fits whole or is refused whole. Feed it the batch in
    // order as (sequence, count) runs; a sequence may come back in later runs.
    // Allocation-free: per-sequence and per-block scratch stamped with a fresh
    // epoch, so one count never sees another's.
    struct Demand {
        pkv_block_manager& bm;
        const uint64_t epoch;
        int64_t blocks = 0, cows = 0;

        explicit Demand(pkv_block_manager& m) : bm(m), epoch(++m.epoch) {}

        void add(Seq& s, int64_t k) {
            if (k <= 0) return;
            const int64_t bs = bm.block_size;
            const bool touched = s.demand_epoch == epoch;
            const int64_t L = touched ? s.demand_len : s.len;
            // A sequence's first append into a partial last block copies it
            // when another table still holds it; later ones write in place.
            if (!touched && L % bs != 0) {
                const int32_t last = s.table.back();
                if (bm.drop_epoch[last] != epoch) {
                    bm.drop_epoch[last] = epoch;
                    bm.drop_count[last] = 0;
                }
                if (bm.ref[last] - bm.drop_count[last] > 1) {
                    blocks += 1;
                    cows += 1;
                    bm.drop_count[last] += 1;
                }
            }
            blocks += (L + k + bs - 1) / bs - (L + bs - 1) / bs;   // block starts in [L, L+k)
            s.demand_epoch = epoch;
            s.demand_len = L + k;
        }

        bool fits() const { return blocks <= (int64_t)bm.device_available(); }
    };
};

extern "C" {

pkv_block_manager* bm_create(int num_blocks, int block_size, const int32_t* free_order,
                             int num_free) {
    if (num_blocks <= 0 || block_size <= 0 || num_free < 0 || num_free > num_blocks ||
        (num_free > 0 && free_order == nullptr))
        return nullptr;
    auto* bm = new (std::nothrow) pkv_block_manager();
    if (!bm) return nullptr;
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->ref.assign(num_blocks, 0);
    bm->drop_epoch.assign(num_blocks, 0);
    bm->drop_count.assign(num_blocks, 0);
    std::vector<char> seen(num_blocks, 0);
    for (int i = 0; i < num_free; ++i) {
        const int32_t b = free_order[i];
        if (b < 0 || b >= num_blocks || seen[b]) {
            delete bm;
            return nullptr;
        }
        seen[b] = 1;
        bm->free_list.push_back(b);
    }
    return bm;
}

void bm_destroy(pkv_block_manager* bm) { delete bm; }

int bm_add_seq(pkv_block_manager* bm, int64_t seq_id) {
    if (!bm) return PKV_ERR_INVALID_ARG;
    if (bm->seqs.count(seq_id)) return PKV_ERR_INVALID_ARG;
    bm->seqs.emplace(seq_id, pkv_block_manager::Seq{});
    return PKV_OK;
}

int bm_append_slot(pkv_block_manager* bm, int64_t seq_id, int64_t* slot, int32_t* cow_src,
                   int32_t* cow_dst) {
    if (!bm || !slot || !cow_src || !cow_dst) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
    return bm->append(it->second, slot, cow_src, cow_dst);
}

int bm_append_n(pkv_block_manager* bm, int64_t seq_id, int n, int64_t* cow_pairs, int cow_cap,
                int* num_cow) {
    if (!bm || n < 0 || !num_cow || (cow_cap > 0 && !cow_pairs)) return PKV_ERR_INVALID_ARG;
    *num_cow = 0;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
    if (it->second.swapped) return PKV_ERR_INVALID_ARG;
    pkv_block_manager::Demand need(*bm);
    need.add(it->second, n);
    if (need.cows > cow_cap) return PKV_ERR_INVALID_ARG;
    if (!need.fits()) return PKV_ERR_POOL_EXHAUSTED;
    for (int i = 0; i < n; ++i) {
        int64_t slot;
        int32_t src, dst;
        const int st = bm->append(it->second, &slot, &src, &dst);
        if (st != PKV_OK) return st;                   // cannot happen after the checks
        if (src >= 0) {
            cow_pairs[2 * *num_cow] = src;
            cow_pairs[2 * *num_cow + 1] = dst;
            *num_cow += 1;
        }
    }
    return PKV_OK;
}

int bm_append_slots(pkv_block_manager* bm, const int64_t* seq_ids, int n, int64_t* slots,
                    int64_t* cow_pairs, int* num_cow) {
    if (!bm || n < 0 || (n > 0 && (!seq_ids || !slots || !cow_pairs)) || !num_cow)
        return PKV_ERR_INVALID_ARG;
    *num_cow = 0;
    std::vector<pkv_block_manager::Seq*> seqs(n);
    pkv_block_manager::Demand need(*bm);
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
        if (it->second.swapped) return PKV_ERR_INVALID_ARG;
        seqs[i] = &it->second;
        need.add(it->second, 1);
    }
    if (!need.fits()) return PKV_ERR_POOL_EXHAUSTED;
    for (int i = 0; i < n; ++i) {
        int32_t src, dst;
        const int st = bm->append(*seqs[i], &slots[i], &src, &dst);
        if (st != PKV_OK) return st;                   // cannot happen after the checks
        if (src >= 0) {
            cow_pairs[2 * *num_cow] = src;
            cow_pairs[2 * *num_cow + 1] = dst;
            *num_cow += 1;
        }
    }
    return PKV_OK;
}

int bm_fork(pkv_block_manager* bm, int64_t parent, int64_t child) {
    if (!bm) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(parent);
    if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
    if (bm->seqs.count(child) || it->second.swapped) return PKV_ERR_INVALID_ARG;
    pkv_block_manager::Seq c = it->second;    // copy of the parent's table
    for (int32_t b : c.table) bm->ref[b] += 1;
    bm->seqs.emplace(child, std::move(c));
    return PKV_OK;
}

int bm_free_seq(pkv_block_manager* bm, int64_t seq_id) {
    if (!bm) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
    if (it->second.swapped) {
        for (int32_t b : it->second.table) bm->host_free.push_back(b);
    } else {
        bm->release(it->second.table);
    }
    bm->seqs.erase(it);
    return PKV_OK;
}

int bm_beam_step(pkv_block_manager* bm, const int64_t* old_ids, int num_old,
                 const int32_t* parents, const int64_t* new_ids, int num_new) {
    if (!bm || num_old < 0 || num_new < 0 || (num_old > 0 && !old_ids) ||
        (num_new > 0 && (!parents || !new_ids)))
        return PKV_ERR_INVALID_ARG;
    std::unordered_map<int64_t, int> seen;
    seen.reserve((size_t)(num_old + num_new));
    for (int i = 0; i < num_old; ++i) {
        auto it = bm->seqs.find(old_ids[i]);
        if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
        if (it->second.swapped || !seen.emplace(old_ids[i], i).second) return PKV_ERR_INVALID_ARG;
    }
    for (int i = 0; i < num_new; ++i) {
        if (parents[i] < 0 || parents[i] >= num_old) return PKV_ERR_OUT_OF_RANGE;
        if (bm->seqs.count(new_ids[i]) || !seen.emplace(new_ids[i], i).second)
            return PKV_ERR_INVALID_ARG;
    }
    for (int i = 0; i < num_new; ++i) {
        const int st = bm_fork(bm, old_ids[parents[i]], new_ids[i]);
        if (st != PKV_OK) return st;                   // cannot happen after the checks
    }
    for (int i = 0; i < num_old; ++i) {
        const int st = bm_free_seq(bm, old_ids[i]);
        if (st != PKV_OK) return st;
    }
    return PKV_OK;
}

int bm_block_table(const pkv_block_manager* bm, int64_t seq_id, int32_t* out, int cap, int* n) {
    if (!bm || !n || (cap > 0 && !out)) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
    const auto& t = it->second.table;
    *n = (int)t.size();
    for (int i = 0; i < *n && i < cap; ++i) out[i] = t[i];
    return (int)t.size() <= cap ? PKV_OK : PKV_ERR_INVALID_ARG;
}

int bm_build_tables(const pkv_block_manager* bm, const int64_t* seq_ids, int n, int max_blocks,
                    int32_t* tables, int32_t* seq_lens) {
    if (!bm || n < 0 || max_blocks < 0 || (n > 0 && (!seq_ids || !seq_lens)) ||
        (n > 0 && max_blocks > 0 && !tables))
        return PKV_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
        const auto& s = it->second;
        if ((int64_t)s.table.size() > max_blocks || s.len > INT32_MAX || s.swapped)
            return PKV_ERR_INVALID_ARG;
        int32_t* row = tables + (size_t)i * max_blocks;
        std::fill(std::copy(s.table.begin(), s.table.end(), row), row + max_blocks, -1);
        seq_lens[i] = (int32_t)s.len;
    }
    return PKV_OK;
}

int bm_seq_len(const pkv_block_manager* bm, int64_t seq_id, int* len) {
    if (!bm || !len) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
    *len = (int)it->second.len;
    return PKV_OK;
}

int bm_refcount(const pkv_block_manager* bm, int block, int* count) {
    if (!bm || !count) return PKV_ERR_INVALID_ARG;
    if (block < 0 || block >= bm->num_blocks) return PKV_ERR_OUT_OF_RANGE;
    *count = bm->ref[block];
    return PKV_OK;
}

int bm_num_free(const pkv_block_manager* bm) { return bm ? (int)bm->free_list.size() : -1; }

// Sequences that point at the same physical blocks (forks of one prompt) can
// share the attention work on those blocks, not only their memory: group them
// by their first block, and take as each group's prefix the leading block ids
// all members have in common, up to the blocks every member has filled.
int bm_prefix_groups(const pkv_block_manager* bm, const int64_t* seq_ids, int n, int max_members,
                     int32_t* group_members, int32_t* group_prefix, int32_t* seq_group,
                     int32_t* group_blocks, int* num_groups) {
    if (!bm || n < 0 || max_members < 1 || !num_groups ||
        (n > 0 && (!seq_ids || !group_members || !group_prefix || !seq_group)))
        return PKV_ERR_INVALID_ARG;
    *num_groups = 0;
    std::vector<const pkv_block_manager::Seq*> seqs(n);
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
        if (it->second.swapped) return PKV_ERR_INVALID_ARG;
        seqs[i] = &it->second;
        seq_group[i] = -1;
    }
    // Buckets of batch indices by first block, each in batch order, the buckets
    // in order of their first member: (block, index) pairs sorted, then the
    // runs of equal blocks sorted by their first index.
    std::vector<std::pair<int32_t, int>> by_block;
    by_block.reserve((size_t)n);
    for (int i = 0; i < n; ++i)
        if (!seqs[i]->table.empty()) by_block.emplace_back(seqs[i]->table[0], i);
    std::sort(by_block.begin(), by_block.end());
    struct Run { int first; size_t a, b; };
    std::vector<Run> runs;
    for (size_t a = 0, b; a < by_block.size(); a = b) {
        for (b = a + 1; b < by_block.size() && by_block[b].first == by_block[a].first; ++b) {}
        runs.push_back({by_block[a].second, a, b});
    }
    std::sort(runs.begin(), runs.end(), [](const Run& x, const Run& y) { return x.first < y.first; });
    std::vector<int> mem;
    int ng = 0;
    for (const Run& r : runs) {
        mem.clear();
        for (size_t j = r.a; j < r.b; ++j) mem.push_back(by_block[j].second);
        for (size_t c = 0; c < mem.size(); c += (size_t)max_members) {
            const size_t e = std::min(mem.size(), c + (size_t)max_members);
            if (e - c < 2) continue;
            int64_t full = INT64_MAX;                // blocks every member has filled
            for (size_t k = c; k < e; ++k)
                full = std::min<int64_t>(full, seqs[mem[k]]->len / bm->block_size);
            const auto& t0 = seqs[mem[c]]->table;
            int64_t prefix = 0;
            while (prefix < full) {
                bool same = true;
                for (size_t k = c + 1; k < e && same; ++k)
                    same = seqs[mem[k]]->table[prefix] == t0[prefix];
                if (!same) break;
                ++prefix;
            }
            if (prefix < 1) continue;
            int32_t* row = group_members + (size_t)ng * max_members;
            for (int k = 0; k < max_members; ++k)
                row[k] = c + k < e ? (int32_t)mem[c + k] : -1;
            group_prefix[ng] = (int32_t)prefix;
            if (group_blocks) {                      // the shared blocks once, then each own tail
                int64_t list = prefix;
                for (size_t k = c; k < e; ++k)
                    list += (seqs[mem[k]]->len + bm->block_size - 1) / bm->block_size - prefix;
                group_blocks[ng] = (int32_t)std::min<int64_t>(list, INT32_MAX);
            }
            for (size_t k = c; k < e; ++k) seq_group[mem[k]] = ng;
            ++ng;
        }
    }
    *num_groups = ng;
    return PKV_OK;
}

int bm_plan_decode(pkv_block_manager* bm, const int64_t* seq_ids, int n, int max_blocks,
                   int64_t* slots, int64_t* cow_pairs, int* num_cow, int32_t* tables,
                   int32_t* seq_lens, int max_members, int32_t* group_members,
                   int32_t* group_prefix, int32_t* seq_group, int32_t* group_blocks,
                   int32_t* ungrouped, int* num_groups, int* num_ungrouped,
                   int* max_group_blocks) {
    if (!bm || n < 0 || max_blocks < 0 || !num_cow)
        return PKV_ERR_INVALID_ARG;
    const bool groups = max_members >= 1;
    if (groups && (!ungrouped || !group_blocks || !num_groups || !num_ungrouped ||
                   !max_group_blocks))
        return PKV_ERR_INVALID_ARG;
    // every table must still fit max_blocks after its append: checked before any
    // append, so a refusal changes nothing
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
        const auto& sq = it->second;
        const int64_t after = (int64_t)sq.table.size() + (sq.len % bm->block_size == 0 ? 1 : 0);
        if (after > max_blocks) return PKV_ERR_INVALID_ARG;
    }
    int st = bm_append_slots(bm, seq_ids, n, slots, cow_pairs, num_cow);
    if (st != PKV_OK) return st;
    st = bm_build_tables(bm, seq_ids, n, max_blocks, tables, seq_lens);
    if (st != PKV_OK) return st;
    if (!groups) return PKV_OK;
    st = bm_prefix_groups(bm, seq_ids, n, max_members, group_members, group_prefix, seq_group,
                          group_blocks, num_groups);
    if (st != PKV_OK) return st;
    int nu = 0, mgb = 0;
    for (int i = 0; i < n; ++i)
        if (seq_group[i] < 0) ungrouped[nu++] = i;
    for (int g = 0; g < *num_groups; ++g) mgb = std::max(mgb, (int)group_blocks[g]);
    *num_ungrouped = nu;
    *max_group_blocks = mgb;
    return PKV_OK;
}

int bm_enable_prefix_caching(pkv_block_manager* bm) {
    if (!bm || !bm->seqs.empty()) return PKV_ERR_INVALID_ARG;
    if (bm->caching) return PKV_OK;
    bm->caching = true;
    bm->registered.assign(bm->num_blocks, 0);
    bm->key_hash.assign(bm->num_blocks, 0);
    bm->parent_hash.assign(bm->num_blocks, 0);
    bm->block_tokens.assign((size_t)bm->num_blocks * bm->block_size, kUnknownToken);
    bm->ev_pos.resize(bm->num_blocks);
    bm->in_ev.assign(bm->num_blocks, 0);
    return PKV_OK;
}

int bm_add_seq_prompt(pkv_block_manager* bm, int64_t seq_id, const int32_t* prompt, int n,
                      int* num_cached) {
    if (!bm || !bm->caching || n < 0 || (n > 0 && !prompt) || !num_cached)
        return PKV_ERR_INVALID_ARG;
    if (bm->seqs.count(seq_id)) return PKV_ERR_INVALID_ARG;
    pkv_block_manager::Seq s;
    const int bs = bm->block_size;
    const int reusable = n > 0 ? (n - 1) / bs : 0;
    std::vector<int64_t> tok(prompt, prompt + n);
    uint64_t h = kPrefixSeed;
    for (int i = 0; i < reusable; ++i) {
        const uint64_t key = chain(h, tok.data() + (size_t)i * bs, bs);
        bm->lookup_blocks += 1;
        const int32_t b = bm->find(h, key, tok.data() + (size_t)i * bs);
        if (b < 0) break;
        bm->hit_blocks += 1;
        if (bm->ref[b] == 0 && bm->in_ev[b]) {      // revive
            bm->evictable.erase(bm->ev_pos[b]);
            bm->in_ev[b] = 0;
        }
        bm->ref[b] += 1;
        s.table.push_back(b);
        s.hashes.push_back(key);
        h = key;
    }
    s.len = (int64_t)s.table.size() * bs;
    s.tokens.assign(tok.begin(), tok.begin() + s.len);
    *num_cached = (int)s.len;
    bm->seqs.emplace(seq_id, std::move(s));
    return PKV_OK;
}

int bm_append_tokens(pkv_block_manager* bm, int64_t seq_id, const int32_t* tokens, int n,
                     int64_t* slots, int64_t* cow_pairs, int cow_cap, int* num_cow) {
    if (!bm || n < 0 || (n > 0 && (!tokens || !slots)) || !num_cow || (cow_cap > 0 && !cow_pairs))
        return PKV_ERR_INVALID_ARG;
    *num_cow = 0;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
    if (it->second.swapped) return PKV_ERR_INVALID_ARG;
    pkv_block_manager::Demand need(*bm);
    need.add(it->second, n);
    if (need.cows > cow_cap) return PKV_ERR_INVALID_ARG;
    if (!need.fits()) return PKV_ERR_POOL_EXHAUSTED;
    for (int i = 0; i < n; ++i) {
        int32_t src, dst;
        const int st = bm->append(it->second, (int64_t)tokens[i], &slots[i], &src, &dst);
        if (st != PKV_OK) return st;                   // cannot happen after the checks
        if (src >= 0) {
            cow_pairs[2 * *num_cow] = src;
            cow_pairs[2 * *num_cow + 1] = dst;
            *num_cow += 1;
        }
    }
    return PKV_OK;
}

int bm_cache_stats(const pkv_block_manager* bm, int64_t* hit_blocks, int64_t* lookup_blocks,
                   int* num_cached, int* num_evictable) {
    if (!bm || !hit_blocks || !lookup_blocks || !num_cached || !num_evictable)
        return PKV_ERR_INVALID_ARG;
    *hit_blocks = bm->hit_blocks;
    *lookup_blocks = bm->lookup_blocks;
    *num_cached = (int)bm->index.size();
    *num_evictable = (int)bm->evictable.size();
    return PKV_OK;
}

int bm_evictable_list(const pkv_block_manager* bm, int32_t* out, int cap) {
    if (!bm) return -1;
    int i = 0;
    for (int32_t b : bm->evictable) {
        if (i < cap && out) out[i] = b;
        ++i;
    }
    return i;
}

int bm_set_host_blocks(pkv_block_manager* bm, int num_host_blocks) {
    if (!bm || num_host_blocks < 0 || !bm->seqs.empty()) return PKV_ERR_INVALID_ARG;
    bm->num_host_blocks = num_host_blocks;
    bm->host_free.clear();
    for (int i = 0; i < num_host_blocks; ++i) bm->host_free.push_back(i);
    return PKV_OK;
}

int bm_swap_out(pkv_block_manager* bm, int64_t seq_id, int64_t* pairs, int cap, int* num_pairs) {
    if (!bm || !num_pairs || (cap > 0 && !pairs)) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
    auto& s = it->second;
    *num_pairs = (int)s.table.size();
    if (s.swapped || cap < (int)s.table.size()) return PKV_ERR_INVALID_ARG;
    if (s.table.size() > bm->host_free.size()) return PKV_ERR_POOL_EXHAUSTED;
    std::vector<int32_t> host(s.table.size());
    for (size_t i = 0; i < host.size(); ++i) {
        host[i] = bm->host_free.front();
        bm->host_free.pop_front();
        pairs[2 * i] = s.table[i];
        pairs[2 * i + 1] = host[i];
    }
    bm->release(s.table);
    s.table = std::move(host);
    s.swapped = true;
    return PKV_OK;
}

int bm_swap_in(pkv_block_manager* bm, int64_t seq_id, int64_t* pairs, int cap, int* num_pairs) {
    if (!bm || !num_pairs || (cap > 0 && !pairs)) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
    auto& s = it->second;
    *num_pairs = (int)s.table.size();
    if (!s.swapped || cap < (int)s.table.size()) return PKV_ERR_INVALID_ARG;
    if (s.table.size() > bm->device_available()) return PKV_ERR_POOL_EXHAUSTED;
    for (size_t i = 0; i < s.table.size(); ++i) {
        const int32_t h = s.table[i];
        const int32_t d = bm->take();
        pairs[2 * i] = h;
        pairs[2 * i + 1] = d;
        s.table[i] = d;
        bm->host_free.push_back(h);
    }
    s.swapped = false;
    return PKV_OK;
}

int bm_is_swapped(const pkv_block_manager* bm, int64_t seq_id, int* swapped) {
    if (!bm || !swapped) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
    *swapped = it->second.swapped ? 1 : 0;
    return PKV_OK;
}

int bm_host_free_list(const pkv_block_manager* bm, int32_t* out, int cap) {
    if (!bm) return -1;
    int i = 0;
    for (int32_t b : bm->host_free) {
        if (i < cap && out) out[i] = b;
        ++i;
    }
    return i;
}

int bm_free_list(const pkv_block_manager* bm, int32_t* out, int cap) {
    if (!bm) return -1;
    int i = 0;
    for (int32_t b : bm->free_list) {
        if (i < cap && out) out[i] = b;
        ++i;
    }
    return i;
}

}  // extern "C"
