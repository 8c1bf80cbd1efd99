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
//
// Prefix caching ("PagedAttention por dentro", section "Prefix caching
// cross-session"; "Cómo funciona realmente vLLM", section "Automatic Prefix
// Caching"): full blocks whose K/V are written can be indexed by a key that
// hashes their content and everything before it,
//     key_j = FNV1a64(le64(key_{j-1}) || le32(tokens of block j)), key_{-1} = 0,
// and a new sequence that begins with the same tokens reuses them.  A lookup
// also compares the block's own tokens.  Released blocks that carry a key wait
// in an evictable list (oldest release first) and are handed out only when the
// free list is empty, losing their key then.
#include <cstdint>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

namespace {

constexpr uint64_t kFnvOffset = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;

uint64_t fnv1a_bytes(uint64_t h, const uint8_t *p, size_t n) {
    for (size_t i = 0; i < n; ++i) {
        h ^= p[i];
        h *= kFnvPrime;
    }
    return h;
}

uint64_t block_key(uint64_t parent, const int32_t *tokens, int block_size) {
    uint8_t buf[8];
    for (int i = 0; i < 8; ++i) buf[i] = (uint8_t)(parent >> (8 * i));
    uint64_t h = fnv1a_bytes(kFnvOffset, buf, 8);
    for (int t = 0; t < block_size; ++t) {
        const uint32_t v = (uint32_t)tokens[t];
        uint8_t b4[4] = {(uint8_t)v, (uint8_t)(v >> 8), (uint8_t)(v >> 16), (uint8_t)(v >> 24)};
        h = fnv1a_bytes(h, b4, 4);
    }
    return h;
}

}  // namespace

struct pa_bm {
    int num_blocks;
    int block_size;
    std::vector<int32_t> free_stack;   // back() is handed out next
    std::vector<int32_t> ref;
    struct Seq {
        std::vector<int32_t> table;   // -1: released by a window trim; -2: swapped out
        int64_t tokens = 0;
        bool swapped = false;
    };
    std::unordered_map<int, Seq> seqs;
    // prefix cache
    std::unordered_map<uint64_t, int32_t> cached;       // key -> block
    std::vector<uint8_t> has_key;
    std::vector<uint64_t> key_of;
    std::vector<std::vector<int32_t>> tokens_of;       // a keyed block's own tokens
    std::list<int32_t> evictable;                       // front = oldest release
    std::vector<std::list<int32_t>::iterator> ev_pos;
    std::vector<uint8_t> in_ev;

    size_t available() const { return free_stack.size() + evictable.size(); }

    int32_t take() {
        int32_t b;
        if (!free_stack.empty()) {
            b = free_stack.back();
            free_stack.pop_back();
        } else {
            b = evictable.front();
            evictable.pop_front();
            in_ev[b] = 0;
            cached.erase(key_of[b]);
            has_key[b] = 0;
            tokens_of[b].clear();
        }
        ref[b] = 1;
        return b;
    }
    void release(int32_t b) {
        ref[b] -= 1;
        if (ref[b] == 0) {
            if (has_key[b]) {
                ev_pos[b] = evictable.insert(evictable.end(), b);
                in_ev[b] = 1;
            } else {
                free_stack.push_back(b);
            }
        }
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
    bm->has_key.assign((size_t)num_blocks, 0);
    bm->key_of.assign((size_t)num_blocks, 0);
    bm->tokens_of.resize((size_t)num_blocks);
    bm->ev_pos.resize((size_t)num_blocks);
    bm->in_ev.assign((size_t)num_blocks, 0);
    bm->free_stack.reserve((size_t)num_blocks);
    for (int b = num_blocks - 1; b >= 0; --b) bm->free_stack.push_back(b);
    return bm;
}

extern "C" void pa_bm_destroy(pa_bm *bm) { delete bm; }

extern "C" pa_status pa_bm_alloc_seq(pa_bm *bm, int seq, int num_tokens) {
    if (bm == nullptr || num_tokens < 0) return PA_ERR_INVALID_ARG;
    if (bm->seqs.count(seq)) return PA_ERR_NOT_FOUND;
    const int64_t need = bm->blocks_for(num_tokens);
    if (need > (int64_t)bm->available()) return PA_ERR_NO_BLOCKS;
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
    if (it->second.swapped) return PA_ERR_INVALID_ARG;
    pa_bm::Seq s = it->second;
    for (int32_t b : s.table)
        if (b >= 0) bm->ref[b] += 1;   // -1: released by pa_bm_trim_window
    bm->seqs.emplace(child, std::move(s));
    return PA_OK;
}

static pa_status make_private(pa_bm *bm, pa_bm::Seq &s, int logical, int32_t *src, int32_t *dst) {
    const int32_t old = s.table[(size_t)logical];
    if (old < 0) return PA_ERR_INVALID_ARG;   // released by pa_bm_trim_window
    if (bm->ref[old] <= 1) {
        // Already private.  A block indexed by the prefix cache is about to be
        // written in place, so its content will no longer match its key: the
        // key is dropped and a later lookup cannot hand the block out.
        if (bm->has_key[old]) {
            bm->cached.erase(bm->key_of[old]);
            bm->has_key[old] = 0;
            bm->tokens_of[old].clear();
        }
        *src = -1;
        *dst = -1;
        return PA_OK;
    }
    if (bm->available() == 0) return PA_ERR_NO_BLOCKS;
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
    if (logical_block < 0 || (size_t)logical_block >= it->second.table.size() ||
        it->second.swapped)
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
    if (s.swapped) return PA_ERR_INVALID_ARG;
    const int64_t n = s.tokens;
    int32_t src = -1, dst = -1;
    if (n % bm->block_size == 0) {
        if (bm->available() == 0) return PA_ERR_NO_BLOCKS;
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
    for (size_t i = t.size(); i-- > 0;)
        if (t[i] >= 0) bm->release(t[i]);
    bm->seqs.erase(it);
    return PA_OK;
}

// Sliding window ("PagedAttention por dentro", section "Sliding window
// attention": the engine keeps only the blocks of the active window and frees
// the older ones).  A sequence of N tokens that attends to its last `window`
// tokens never reads a block whose positions all lie before N - window: those
// are released (last such entry first) and their table entries become -1.
extern "C" int pa_bm_trim_window(pa_bm *bm, int seq, int window) {
    if (bm == nullptr || window <= 0) return -1;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return -1;
    pa_bm::Seq &s = it->second;
    if (s.swapped) return -1;
    const int64_t dead = s.tokens > window ? (s.tokens - window) / bm->block_size : 0;
    int released = 0;
    for (int64_t j = dead; j-- > 0;) {
        const int32_t b = s.table[(size_t)j];
        if (b < 0) continue;
        bm->release(b);
        s.table[(size_t)j] = -1;
        ++released;
    }
    return released;
}

extern "C" int pa_bm_num_evictable(const pa_bm *bm) {
    return bm == nullptr ? -1 : (int)bm->evictable.size();
}

extern "C" pa_status pa_bm_alloc_seq_cached(pa_bm *bm, int seq, const int32_t *tokens,
                                            int num_tokens, int *num_cached_tokens) {
    if (bm == nullptr || num_tokens < 0 || num_cached_tokens == nullptr ||
        (num_tokens > 0 && tokens == nullptr))
        return PA_ERR_INVALID_ARG;
    if (bm->seqs.count(seq)) return PA_ERR_NOT_FOUND;
    std::vector<int32_t> hits;
    uint64_t parent = 0;
    const int bs = bm->block_size;
    for (int j = 0; j < num_tokens / bs; ++j) {
        const int32_t *own = tokens + (size_t)j * bs;
        parent = block_key(parent, own, bs);
        auto f = bm->cached.find(parent);
        if (f == bm->cached.end()) break;
        const std::vector<int32_t> &stored = bm->tokens_of[f->second];
        bool same = true;
        for (int k = 0; k < bs && same; ++k) same = stored[k] == own[k];
        if (!same) break;
        hits.push_back(f->second);
    }
    const int64_t need = bm->blocks_for(num_tokens) - (int64_t)hits.size();
    int64_t reusable = 0;
    for (int32_t b : hits) reusable += bm->ref[b] == 0 ? 1 : 0;
    if (need > (int64_t)bm->available() - reusable) return PA_ERR_NO_BLOCKS;
    for (int32_t b : hits) {
        if (bm->ref[b] == 0) {
            bm->evictable.erase(bm->ev_pos[b]);
            bm->in_ev[b] = 0;
        }
        bm->ref[b] += 1;
    }
    pa_bm::Seq s;
    s.tokens = num_tokens;
    s.table = hits;
    for (int64_t i = 0; i < need; ++i) s.table.push_back(bm->take());
    bm->seqs.emplace(seq, std::move(s));
    *num_cached_tokens = (int)hits.size() * bs;
    return PA_OK;
}

extern "C" int pa_bm_register_prefix(pa_bm *bm, int seq, const int32_t *tokens, int num_tokens) {
    if (bm == nullptr || num_tokens < 0 || (num_tokens > 0 && tokens == nullptr)) return -1;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end() || it->second.swapped) return -1;
    const std::vector<int32_t> &table = it->second.table;
    const int bs = bm->block_size;
    const int64_t n = num_tokens < it->second.tokens ? num_tokens : it->second.tokens;
    int added = 0;
    uint64_t parent = 0;
    for (int64_t j = 0; j < n / bs; ++j) {
        const int32_t *own = tokens + (size_t)j * bs;
        parent = block_key(parent, own, bs);
        const int32_t b = table[(size_t)j];
        if (b < 0 || bm->cached.count(parent) || bm->has_key[b]) continue;
        bm->cached.emplace(parent, b);
        bm->has_key[b] = 1;
        bm->key_of[b] = parent;
        bm->tokens_of[b].assign(own, own + bs);
        ++added;
    }
    return added;
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
        if (it->second.table.size() > (size_t)max_blocks || it->second.swapped)
            return PA_ERR_INVALID_ARG;
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

extern "C" pa_status pa_bm_swap_out(pa_bm *bm, int seq, int32_t *block_ids, int cap,
                                    int *num_ids) {
    if (bm == nullptr || num_ids == nullptr || cap < 0 || (cap > 0 && block_ids == nullptr))
        return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
    pa_bm::Seq &s = it->second;
    if (s.swapped) return PA_ERR_INVALID_ARG;
    int n = 0;
    for (int32_t b : s.table) n += b >= 0;
    if (n > cap) return PA_ERR_INVALID_ARG;
    int k = 0;
    for (int32_t b : s.table)
        if (b >= 0) block_ids[k++] = b;
    for (size_t i = s.table.size(); i-- > 0;) {
        if (s.table[i] < 0) continue;
        bm->release(s.table[i]);
        s.table[i] = -2;
    }
    s.swapped = true;
    *num_ids = n;
    return PA_OK;
}

extern "C" pa_status pa_bm_swap_in(pa_bm *bm, int seq, int32_t *block_ids, int cap, int *num_ids) {
    if (bm == nullptr || num_ids == nullptr || cap < 0 || (cap > 0 && block_ids == nullptr))
        return PA_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PA_ERR_NOT_FOUND;
    pa_bm::Seq &s = it->second;
    if (!s.swapped) return PA_ERR_INVALID_ARG;
    int n = 0;
    for (int32_t b : s.table) n += b == -2;
    if (n > cap) return PA_ERR_INVALID_ARG;
    if ((size_t)n > bm->available()) return PA_ERR_NO_BLOCKS;
    int k = 0;
    for (int32_t &b : s.table)
        if (b == -2) {
            b = bm->take();
            block_ids[k++] = b;
        }
    s.swapped = false;
    *num_ids = n;
    return PA_OK;
}

// Occupancy and internal fragmentation of the pool ("Cómo funciona realmente
// vLLM", section "La sobre-reserva estática y los tres tipos de desperdicio":
// internal fragmentation is reserved slots that never receive a token; with
// 16-token blocks only each sequence's last block can hold such slots).  A
// block's filled slots are the longest run any table entry pointing at it has
// written: every entry fills a block from offset 0 up.
extern "C" pa_status pa_bm_stats(const pa_bm *bm, pa_bm_stats_t *out) {
    if (bm == nullptr || out == nullptr) return PA_ERR_INVALID_ARG;
    const int64_t bs = bm->block_size;
    std::vector<int32_t> fill((size_t)bm->num_blocks, 0);
    int64_t logical = 0;
    for (const auto &kv : bm->seqs) {
        const pa_bm::Seq &s = kv.second;
        for (size_t j = 0; j < s.table.size(); ++j) {
            const int32_t b = s.table[j];
            if (b < 0) continue;   // released by a window trim, or swapped out
            const int64_t left = s.tokens - (int64_t)j * bs;
            const int32_t f = (int32_t)(left < bs ? left : bs);
            logical += f;
            if (f > fill[(size_t)b]) fill[(size_t)b] = f;
        }
    }
    int64_t used = 0, shared = 0, filled = 0;
    for (int b = 0; b < bm->num_blocks; ++b) {
        used += bm->ref[(size_t)b] >= 1;
        shared += bm->ref[(size_t)b] >= 2;
        filled += fill[(size_t)b];
    }
    out->num_blocks = bm->num_blocks;
    out->free_blocks = (int64_t)bm->free_stack.size();
    out->evictable_blocks = (int64_t)bm->evictable.size();
    out->used_blocks = used;
    out->shared_blocks = shared;
    out->reserved_slots = used * bs;
    out->filled_slots = filled;
    out->logical_tokens = logical;
    out->internal_fragmentation =
        used == 0 ? 0.0 : (double)(used * bs - filled) / (double)(used * bs);
    return PA_OK;
}
