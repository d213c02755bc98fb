// Host-side block manager for the paged KV cache: pool, block tables, reference
// counts with copy-on-write, prefix cache with exact matching, LRU eviction.
// The C ABI and the policy it follows are documented in include/pa_blocks.h.
#include <stdio.h>
#include <string.h>

#include <list>
#include <string>
#include <unordered_map>
#include <vector>

#include "pa_blocks.h"

namespace pa {
pa_status fail(pa_status status, const char *fmt, ...);
}

namespace {

struct Sequence {
    std::vector<int32_t> blocks;  // logical block j -> physical block
    int64_t len = 0;              // tokens written
    uint64_t chain = 0;           // prefix-cache node of the last full block (0: none yet)
    bool ids_known = true;        // every token so far came with its id
    std::vector<int32_t> pending; // ids of the tokens in the current partial block
};

}  // namespace

struct pa_block_manager {
    int N = 0, bs = 0;
    std::vector<int32_t> refcnt;   // holders per block
    std::vector<int32_t> fill;     // token slots written in the block
    std::vector<uint64_t> node;    // prefix-cache node id of a registered block, else 0
    std::vector<std::string> key;  // its registry key
    std::vector<int32_t> free_stack;
    std::list<int32_t> lru;        // registered blocks nobody holds; front = oldest
    std::vector<std::list<int32_t>::iterator> lru_pos;
    std::vector<char> in_lru;
    // registry: (parent node, the block's token ids) -> physical block; a flattened
    // prefix trie whose edges are whole blocks
    std::unordered_map<std::string, int32_t> registry;
    std::unordered_map<int64_t, Sequence> seqs;
    uint64_t next_node = 1;
    pa_bm_stats st{};

    static std::string make_key(uint64_t parent, const int32_t *ids, int n) {
        std::string k(sizeof(uint64_t) + sizeof(int32_t) * (size_t)n, '\0');
        memcpy(&k[0], &parent, sizeof(uint64_t));
        memcpy(&k[sizeof(uint64_t)], ids, sizeof(int32_t) * (size_t)n);
        return k;
    }

    int64_t available() const { return (int64_t)free_stack.size() + (int64_t)lru.size(); }

    void unregister(int32_t b) {
        if (node[b] != 0) {
            auto it = registry.find(key[b]);
            if (it != registry.end() && it->second == b) registry.erase(it);
            node[b] = 0;
            key[b].clear();
        }
    }

    // A block for new content: the free list first, then the oldest cached block.
    int32_t take() {
        int32_t b;
        if (!free_stack.empty()) {
            b = free_stack.back();
            free_stack.pop_back();
        } else {
            b = lru.front();
            lru.pop_front();
            in_lru[b] = 0;
            unregister(b);
            ++st.evictions;
        }
        refcnt[b] = 1;
        fill[b] = 0;
        return b;
    }

    void hold(int32_t b) {
        if (in_lru[b]) {
            lru.erase(lru_pos[b]);
            in_lru[b] = 0;
        }
        ++refcnt[b];
    }

    void release(int32_t b) {
        if (--refcnt[b] > 0) return;
        if (node[b] != 0) {
            lru.push_back(b);
            lru_pos[b] = std::prev(lru.end());
            in_lru[b] = 1;
        } else {
            free_stack.push_back(b);
        }
    }

    // The sequence's last block just became full: enter it in the prefix registry.
    void register_full(Sequence &s) {
        const int32_t b = s.blocks.back();
        std::string k = make_key(s.chain, s.pending.data(), bs);
        auto it = registry.find(k);
        if (it != registry.end()) {
            s.chain = node[it->second];  // the same prefix is already cached elsewhere
        } else if (node[b] == 0) {
            node[b] = next_node++;
            key[b] = k;
            registry.emplace(std::move(k), b);
            s.chain = node[b];
        } else {
            s.chain = node[b];
        }
        s.pending.clear();
    }
};

using pa::fail;

extern "C" {

pa_status pa_bm_create(int num_blocks, int block_size, pa_block_manager **out) {
    if (!out) return fail(PA_ERR_INVALID_ARG, "pa_bm_create: null output");
    *out = nullptr;
    if (num_blocks <= 0 || block_size <= 0 || block_size > 4096)
        return fail(PA_ERR_INVALID_ARG, "pa_bm_create: num_blocks = %d, block_size = %d", num_blocks,
                    block_size);
    auto *bm = new pa_block_manager();
    bm->N = num_blocks;
    bm->bs = block_size;
    bm->refcnt.assign(num_blocks, 0);
    bm->fill.assign(num_blocks, 0);
    bm->node.assign(num_blocks, 0);
    bm->key.assign(num_blocks, std::string());
    bm->lru_pos.resize(num_blocks);
    bm->in_lru.assign(num_blocks, 0);
    bm->free_stack.reserve(num_blocks);
    for (int b = num_blocks - 1; b >= 0; --b) bm->free_stack.push_back(b);  // block 0 first
    bm->st.num_blocks = num_blocks;
    *out = bm;
    return PA_OK;
}

void pa_bm_destroy(pa_block_manager *bm) { delete bm; }

pa_status pa_bm_add_sequence(pa_block_manager *bm, int64_t seq_id, const int32_t *prompt,
                             int n_prompt, int *n_cached_tokens) {
    if (!bm) return fail(PA_ERR_INVALID_ARG, "pa_bm_add_sequence: null manager");
    if (n_prompt < 0 || (n_prompt > 0 && !prompt))
        return fail(PA_ERR_INVALID_ARG, "pa_bm_add_sequence: bad prompt");
    if (bm->seqs.count(seq_id)) return fail(PA_ERR_INVALID_ARG, "pa_bm_add_sequence: sequence %lld exists", (long long)seq_id);
    Sequence s;
    for (int i = 0; i + bm->bs <= n_prompt; i += bm->bs) {
        ++bm->st.prefix_lookup_blocks;
        auto it = bm->registry.find(pa_block_manager::make_key(s.chain, prompt + i, bm->bs));
        if (it == bm->registry.end()) break;
        const int32_t b = it->second;
        bm->hold(b);
        s.blocks.push_back(b);
        s.len += bm->bs;
        s.chain = bm->node[b];
        ++bm->st.prefix_hit_blocks;
    }
    if (n_cached_tokens) *n_cached_tokens = (int)s.len;
    bm->seqs.emplace(seq_id, std::move(s));
    return PA_OK;
}

pa_status pa_bm_append(pa_block_manager *bm, int64_t seq_id, const int32_t *tokens, int n,
                       int64_t *slots, int64_t *cow, int max_pairs, int *n_cow) {
    if (!bm) return fail(PA_ERR_INVALID_ARG, "pa_bm_append: null manager");
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return fail(PA_ERR_INVALID_ARG, "pa_bm_append: unknown sequence %lld", (long long)seq_id);
    if (n < 0 || (n > 0 && !slots)) return fail(PA_ERR_INVALID_ARG, "pa_bm_append: bad token count or slots");
    if (n_cow) *n_cow = 0;
    if (n == 0) return PA_OK;
    Sequence &s = it->second;
    const int bs = bm->bs;
    const bool need_cow = (s.len % bs) != 0 && bm->refcnt[s.blocks.back()] > 1;
    if (need_cow && (!cow || max_pairs < 1 || !n_cow))
        return fail(PA_ERR_INVALID_ARG, "pa_bm_append: a copy-on-write pair must be returned");
    // blocks this call takes: the copy, plus one per block boundary crossed
    const int64_t first_new = s.len % bs == 0 ? 0 : bs - s.len % bs;  // tokens before a boundary
    const int64_t crossings = n > first_new ? (n - first_new + bs - 1) / bs : 0;
    const int64_t needed = crossings + (need_cow ? 1 : 0);
    if (needed > bm->available())
        return fail(PA_ERR_NO_SPACE, "pa_bm_append: %lld blocks needed, %lld available", (long long)needed,
                    (long long)bm->available());
    if (need_cow) {
        const int32_t src = s.blocks.back();
        const int32_t dst = bm->take();
        bm->fill[dst] = (int32_t)(s.len % bs);
        bm->release(src);
        s.blocks.back() = dst;
        cow[0] = src;
        cow[1] = dst;
        *n_cow = 1;
        ++bm->st.cow_copies;
    }
    if (!tokens) s.ids_known = false;
    for (int i = 0; i < n; ++i) {
        const int off = (int)(s.len % bs);
        if (off == 0) s.blocks.push_back(bm->take());
        const int32_t b = s.blocks.back();
        slots[i] = (int64_t)b * bs + off;
        if (bm->fill[b] < off + 1) bm->fill[b] = off + 1;
        ++s.len;
        if (s.ids_known) {
            s.pending.push_back(tokens[i]);
            if (s.len % bs == 0) bm->register_full(s);
        }
    }
    return PA_OK;
}

pa_status pa_bm_fork(pa_block_manager *bm, int64_t parent_id, int64_t child_id) {
    if (!bm) return fail(PA_ERR_INVALID_ARG, "pa_bm_fork: null manager");
    auto it = bm->seqs.find(parent_id);
    if (it == bm->seqs.end()) return fail(PA_ERR_INVALID_ARG, "pa_bm_fork: unknown sequence %lld", (long long)parent_id);
    if (bm->seqs.count(child_id)) return fail(PA_ERR_INVALID_ARG, "pa_bm_fork: sequence %lld exists", (long long)child_id);
    Sequence child = it->second;
    for (int32_t b : child.blocks) bm->hold(b);
    bm->seqs.emplace(child_id, std::move(child));
    return PA_OK;
}

pa_status pa_bm_free(pa_block_manager *bm, int64_t seq_id) {
    if (!bm) return fail(PA_ERR_INVALID_ARG, "pa_bm_free: null manager");
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return fail(PA_ERR_INVALID_ARG, "pa_bm_free: unknown sequence %lld", (long long)seq_id);
    // last block first: among the cached blocks it releases, the tail of a prefix is
    // the first to be evicted
    const std::vector<int32_t> &blocks = it->second.blocks;
    for (size_t j = blocks.size(); j-- > 0;) bm->release(blocks[j]);
    bm->seqs.erase(it);
    return PA_OK;
}

pa_status pa_bm_block_table(const pa_block_manager *bm, int64_t seq_id, int32_t *table, int capacity,
                            int *n_blocks, int64_t *context_len) {
    if (!bm) return fail(PA_ERR_INVALID_ARG, "pa_bm_block_table: null manager");
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return fail(PA_ERR_INVALID_ARG, "pa_bm_block_table: unknown sequence %lld", (long long)seq_id);
    const Sequence &s = it->second;
    if (n_blocks) *n_blocks = (int)s.blocks.size();
    if (context_len) *context_len = s.len;
    if (table) {
        if (capacity < (int)s.blocks.size())
            return fail(PA_ERR_INVALID_ARG, "pa_bm_block_table: capacity %d < %zu blocks", capacity, s.blocks.size());
        for (size_t j = 0; j < s.blocks.size(); ++j) table[j] = s.blocks[j];
    }
    return PA_OK;
}

pa_status pa_bm_get_stats(const pa_block_manager *bm, pa_bm_stats *out) {
    if (!bm || !out) return fail(PA_ERR_INVALID_ARG, "pa_bm_get_stats: null pointer");
    pa_bm_stats st = bm->st;
    st.free_blocks = (int64_t)bm->free_stack.size();
    st.cached_blocks = (int64_t)bm->lru.size();
    st.used_blocks = 0;
    st.used_slots = 0;
    for (int b = 0; b < bm->N; ++b)
        if (bm->refcnt[b] > 0) {
            ++st.used_blocks;
            st.used_slots += bm->fill[b];
        }
    *out = st;
    return PA_OK;
}

}  // extern "C"
