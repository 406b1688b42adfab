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
#include <algorithm>
#include <climits>
#include <cstdint>
#include <deque>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pagedkv.h"

struct pkv_block_manager {
    int num_blocks = 0;
    int block_size = 0;
    std::deque<int32_t> free_list;       // front = next block handed out
    std::vector<int32_t> ref;            // reference count per physical block
    struct Seq {
        std::vector<int32_t> table;      // logical block i -> physical block id
        int64_t len = 0;                 // tokens cached
    };
    std::unordered_map<int64_t, Seq> seqs;

    int32_t take() {
        int32_t b = free_list.front();
        free_list.pop_front();
        ref[b] = 1;
        return b;
    }

    // One append; on exhaustion nothing changes.
    int append(Seq& s, int64_t* slot, int32_t* cow_src, int32_t* cow_dst) {
        *cow_src = -1;
        *cow_dst = -1;
        const int64_t n = s.len;
        if (n % block_size == 0) {
            if (free_list.empty()) return PKV_ERR_POOL_EXHAUSTED;
            s.table.push_back(take());
        } else {
            const int32_t last = s.table.back();
            if (ref[last] > 1) {                       // shared: copy before writing
                if (free_list.empty()) return PKV_ERR_POOL_EXHAUSTED;
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
        return PKV_OK;
    }
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
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
    *num_cow = 0;
    for (int i = 0; i < n; ++i) {
        int64_t slot;
        int32_t src, dst;
        const int st = bm->append(it->second, &slot, &src, &dst);
        if (st != PKV_OK) return st;
        if (src >= 0) {
            if (*num_cow >= cow_cap) return PKV_ERR_INVALID_ARG;
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
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
        int32_t src, dst;
        const int st = bm->append(it->second, &slots[i], &src, &dst);
        if (st != PKV_OK) return st;
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
    if (bm->seqs.count(child)) return PKV_ERR_INVALID_ARG;
    pkv_block_manager::Seq c = it->second;    // copy of the parent's table
    for (int32_t b : c.table) bm->ref[b] += 1;
    bm->seqs.emplace(child, std::move(c));
    return PKV_OK;
}

int bm_free_seq(pkv_block_manager* bm, int64_t seq_id) {
    if (!bm) return PKV_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
    for (int32_t b : it->second.table) {
        bm->ref[b] -= 1;
        if (bm->ref[b] == 0) bm->free_list.push_back(b);
    }
    bm->seqs.erase(it);
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
        if ((int64_t)s.table.size() > max_blocks || s.len > INT32_MAX) return PKV_ERR_INVALID_ARG;
        int32_t* row = tables + (size_t)i * max_blocks;
        for (int j = 0; j < max_blocks; ++j) row[j] = j < (int)s.table.size() ? s.table[j] : -1;
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
                     int* num_groups) {
    if (!bm || n < 0 || max_members < 1 || !num_groups ||
        (n > 0 && (!seq_ids || !group_members || !group_prefix || !seq_group)))
        return PKV_ERR_INVALID_ARG;
    *num_groups = 0;
    std::vector<const pkv_block_manager::Seq*> seqs(n);
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seq_ids[i]);
        if (it == bm->seqs.end()) return PKV_ERR_OUT_OF_RANGE;
        seqs[i] = &it->second;
        seq_group[i] = -1;
    }
    std::unordered_map<int32_t, std::vector<int>> buckets;
    std::vector<int32_t> order;                      // first blocks in batch order
    for (int i = 0; i < n; ++i) {
        if (seqs[i]->table.empty()) continue;
        const int32_t key = seqs[i]->table[0];
        auto& v = buckets[key];
        if (v.empty()) order.push_back(key);
        v.push_back(i);
    }
    int ng = 0;
    for (int32_t key : order) {
        const std::vector<int>& mem = buckets[key];
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
            for (size_t k = c; k < e; ++k) seq_group[mem[k]] = ng;
            ++ng;
        }
    }
    *num_groups = ng;
    return PKV_OK;
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
