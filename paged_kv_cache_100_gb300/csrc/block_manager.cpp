// Host block manager: the global pool of fixed-size KV blocks, per-sequence
// block tables, reference counts and copy-on-write.
//
// "PagedAttention por dentro: bloques, tabla de páginas, evicción y el estado
// del arte del KV cache en 2026":
//   * "La tabla de páginas (block table)": a sequence that already holds N
//     tokens writes its next token into its last block when N mod 16 != 0 and
//     otherwise appends a block taken from the pool; growing costs one O(1)
//     allocation plus an O(1) append, and freeing returns every block.
//   * "El pool de bloques": one pool shared by all sequences, sized at start.
//   * "Copy-on-write para sampling paralelo": forked sequences share blocks;
//     a sequence about to change a shared block gets its own copy of that
//     block only (the (src, dst) pair goes to pa_block_copy).
//
// Allocation order is deterministic: the free list is a stack that hands out
// 0, 1, 2, ... first, a freed block is the next one handed out, and a table
// is released from its last entry to its first.  Every failing operation
// leaves the manager unchanged.
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

struct pa_bm {
    int num_blocks;
    int block_size;
    std::vector<int32_t> free_stack;   // back() is handed out next
    std::vector<int32_t> ref;
    struct Seq {
        std::vector<int32_t> table;
        int64_t tokens = 0;
    };
    std::unordered_map<int, Seq> seqs;

    int32_t take() {
        const int32_t b = free_stack.back();
        free_stack.pop_back();
        ref[b] = 1;
        return b;
    }
    int64_t blocks_for(int64_t tokens) const { return (tokens + block_size - 1) / block_size; }
};

extern "C" pa_bm *pa_bm_create(int num_blocks, int block_size) {
    if (num_blocks < 0 || block_size <= 0) return nullptr;
    pa_bm *bm = new (std::nothrow) pa_bm();
    if (bm == nullptr) return nullptr;
    bm->num_blocks = num_blocks;
    bm->block_size = block_size;
    bm->ref.assign((size_t)num_blocks, 0);
    bm->free_stack.reserve((size_t)num_blocks);
    for (int b = num_blocks - 1; b >= 0; --b) bm->free_stack.push_back(b);
    return bm;
}

extern "C" void pa_bm_destroy(pa_bm *bm) { delete bm; }

extern "C" pa_status pa_bm_alloc_seq(pa_bm *bm, int seq, int num_tokens) {
    if (bm == nullptr || num_tokens < 0) return PA_ERR_INVALID_ARG;
    if (bm->seqs.count(seq)) return PA_ERR_NOT_FOUND;
    const int64_t need = bm->blocks_for(num_tokens);
    if (need > (int64_t)bm->free_stack.size()) return PA_ERR_NO_BLOCKS;
    pa_bm::Seq s;
    s.tokens = num_tokens;
    s.table.reserve((size_t)need);
    for (int64_t i = 0; i < need; ++i) s.table.push_back(bm->take());
    bm->seqs.emplace(seq, std::move(s));
    return PA_OK;
}

extern "C" pa_status pa_bm_fork(pa_bm *bm, int parent, int child) {
    if (bm == nullptr) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(parent);
    if (it == bm->seqs.end() || bm->seqs.count(child)) return PA_ERR_NOT_FOUND;
    pa_bm::Seq s = it->second;
    for (int32_t b : s.table) bm->ref[b] += 1;
    bm->seqs.emplace(child, std::move(s));
    return PA_OK;
}

static pa_status make_private(pa_bm *bm, pa_bm::Seq &s, int logical, int32_t *src, int32_t *dst) {
    const int32_t old = s.table[(size_t)logical];
    if (bm->ref[old] <= 1) {
        *src = -1;
        *dst = -1;
        return PA_OK;
    }
    if (bm->free_stack.empty()) return PA_ERR_NO_BLOCKS;
    const int32_t fresh = bm->take();
    bm->ref[old] -= 1;
    s.table[(size_t)logical] = fresh;
    *src = old;
    *dst = fresh;
    return PA_OK;
}

extern "C" pa_status pa_bm_make_private(pa_bm *bm, int seq, int logical_block, int32_t *cow_src,
                                        int32_t *cow_dst) {
    if (bm == nullptr || cow_src == nullptr || cow_dst == nullptr) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
    if (logical_block < 0 || (size_t)logical_block >= it->second.table.size())
        return PA_ERR_INVALID_ARG;
    return make_private(bm, it->second, logical_block, cow_src, cow_dst);
}

extern "C" pa_status pa_bm_append_slot(pa_bm *bm, int seq, int64_t *slot, int32_t *cow_src,
                                       int32_t *cow_dst) {
    if (bm == nullptr || slot == nullptr || cow_src == nullptr || cow_dst == nullptr)
        return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
    pa_bm::Seq &s = it->second;
    const int64_t n = s.tokens;
    int32_t src = -1, dst = -1;
    if (n % bm->block_size == 0) {
        if (bm->free_stack.empty()) return PA_ERR_NO_BLOCKS;
        s.table.push_back(bm->take());
    } else {
        pa_status st = make_private(bm, s, (int)s.table.size() - 1, &src, &dst);
        if (st != PA_OK) return st;
    }
    *slot = (int64_t)s.table[(size_t)(n / bm->block_size)] * bm->block_size + n % bm->block_size;
    *cow_src = src;
    *cow_dst = dst;
    s.tokens = n + 1;
    return PA_OK;
}

extern "C" pa_status pa_bm_free_seq(pa_bm *bm, int seq) {
    if (bm == nullptr) return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
    const std::vector<int32_t> &t = it->second.table;
    for (size_t i = t.size(); i-- > 0;) {
        const int32_t b = t[i];
        bm->ref[b] -= 1;
        if (bm->ref[b] == 0) bm->free_stack.push_back(b);
    }
    bm->seqs.erase(it);
    return PA_OK;
}

extern "C" int pa_bm_num_free(const pa_bm *bm) {
    return bm == nullptr ? -1 : (int)bm->free_stack.size();
}

extern "C" int pa_bm_num_tokens(const pa_bm *bm, int seq) {
    if (bm == nullptr) return -1;
    auto it = bm->seqs.find(seq);
    return it == bm->seqs.end() ? -1 : (int)it->second.tokens;
}

extern "C" int pa_bm_ref_count(const pa_bm *bm, int block) {
    if (bm == nullptr || block < 0 || block >= bm->num_blocks) return -1;
    return bm->ref[(size_t)block];
}

extern "C" int pa_bm_table(const pa_bm *bm, int seq, int32_t *out, int cap) {
    if (bm == nullptr) return -1;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return -1;
    const std::vector<int32_t> &t = it->second.table;
    for (int i = 0; i < cap && (size_t)i < t.size(); ++i) out[i] = t[(size_t)i];
    return (int)t.size();
}

extern "C" pa_status pa_bm_append_slots(pa_bm *bm, const int32_t *seqs, int n, int64_t *slots,
                                        int32_t *cow_pairs, int *num_cow, int *num_done) {
    if (bm == nullptr || n < 0 || num_cow == nullptr || num_done == nullptr ||
        (n > 0 && (seqs == nullptr || slots == nullptr || cow_pairs == nullptr)))
        return PA_ERR_INVALID_ARG;
    *num_cow = 0;
    *num_done = 0;
    for (int i = 0; i < n; ++i) {
        int32_t src, dst;
        pa_status st = pa_bm_append_slot(bm, seqs[i], &slots[i], &src, &dst);
        if (st != PA_OK) return st;
        if (src >= 0) {
            cow_pairs[2 * *num_cow] = src;
            cow_pairs[2 * *num_cow + 1] = dst;
            *num_cow += 1;
        }
        *num_done = i + 1;
    }
    return PA_OK;
}

extern "C" pa_status pa_bm_fill_tables(const pa_bm *bm, const int32_t *seqs, int n,
                                       int32_t *tables, int max_blocks, int32_t *context_lens) {
    if (bm == nullptr || n < 0 || max_blocks < 0 ||
        (n > 0 && (seqs == nullptr || tables == nullptr || context_lens == nullptr)))
        return PA_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) {
        auto it = bm->seqs.find(seqs[i]);
        if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
        if (it->second.table.size() > (size_t)max_blocks) return PA_ERR_INVALID_ARG;
    }
    for (int i = 0; i < n; ++i) {
        const pa_bm::Seq &s = bm->seqs.find(seqs[i])->second;
        int32_t *row = tables + (size_t)i * max_blocks;
        size_t j = 0;
        for (; j < s.table.size(); ++j) row[j] = s.table[j];
        for (; j < (size_t)max_blocks; ++j) row[j] = -1;
        context_lens[i] = (int32_t)s.tokens;
    }
    return PA_OK;
}
