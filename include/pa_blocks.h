/*
 * pa_blocks.h -- host-side block manager for the paged KV cache (C ABI).
 *
 * The bookkeeping the source pages describe around the GPU path:
 *   - the cache is a pool of fixed-size physical blocks; each sequence holds a
 *     block table from its logical blocks to physical ones, and only as many blocks
 *     as its current length needs (gotburnout.io "PagedAttention & Gestion du
 *     KV-Cache", section 2 figure; blog.fabienvernieres.com "Cache KV en production",
 *     "PagedAttention : la pagination appliquee au cache KV");
 *   - blocks go back to the common pool as soon as a request ends or is cancelled
 *     (same glossary, section 4, freeing pages on cancellation);
 *   - requests sharing a prefix point at the same physical blocks; a shared block is
 *     copied only when a sequence starts writing its own tokens into it
 *     (copy-on-write, glossary section 3.01), and branches of one request share
 *     their common context (section 3.02);
 *   - prefix caching: full blocks of an already computed prefix are found again by
 *     hashing (gaiatechstar.com forum thread, prefix caching "via un systeme de
 *     hashage"; a chain of block hashes is a prefix trie flattened), reused only when
 *     the prefix tokens are exactly identical (fabienvernieres, "le prefix caching");
 *   - cached blocks no request holds are evicted least-recently-used first when the
 *     pool runs dry (fabienvernieres, "Faire de la place : l'eviction").
 *
 * Policy details fixed here (the pages leave them open): the free list is a stack
 * (the most recently freed block is reused first); a sequence's full blocks are
 * registered in the prefix cache only when token ids are supplied; a block whose
 * last holder leaves goes to the LRU list if it is registered, else to the free
 * list; blocks are taken from the free list first, then by evicting the least
 * recently released cached block.
 *
 * Calls are host-only and not thread-safe (one manager per thread or external
 * locking).  Device copies (copy-on-write pairs, new token slots) are returned to
 * the caller, who passes them to pa_copy_blocks / pa_reshape_and_cache.
 */
#ifndef PA_BLOCKS_H
#define PA_BLOCKS_H

#include <stdint.h>

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_block_manager pa_block_manager;

typedef struct pa_bm_stats {
    int64_t num_blocks;     /* blocks in the pool */
    int64_t free_blocks;    /* on the free list */
    int64_t cached_blocks;  /* held by no sequence, kept for prefix reuse (evictable) */
    int64_t used_blocks;    /* held by at least one sequence */
    int64_t used_slots;     /* token slots written in held blocks, each physical slot once */
    int64_t cow_copies;     /* copy-on-write pairs returned so far */
    int64_t prefix_lookup_blocks; /* full prompt blocks looked up in the prefix cache */
    int64_t prefix_hit_blocks;    /* ... of which were found */
    int64_t evictions;      /* cached blocks reclaimed */
} pa_bm_stats;

/* A manager for a pool of num_blocks blocks of block_size token slots. */
pa_status pa_bm_create(int num_blocks, int block_size, pa_block_manager **out);
void pa_bm_destroy(pa_block_manager *bm);

/*
 * Register sequence seq_id (unique).  With a prompt (token ids, n_prompt > 0) the
 * longest run of leading full blocks whose tokens exactly match a cached prefix is
 * attached to the sequence; *n_cached_tokens (nullable) receives its length (a
 * multiple of the block size; those tokens need no prefill).  The remaining prompt
 * tokens are not appended: the caller appends them with pa_bm_append.
 */
pa_status pa_bm_add_sequence(pa_block_manager *bm, int64_t seq_id, const int32_t *prompt,
                             int n_prompt, int *n_cached_tokens);

/*
 * Append n tokens to a sequence.  slots[i] (n entries) receives the slot of token
 * i: physical block * block_size + offset.  When the sequence's last block is
 * shared with another sequence, it is first copied to a fresh block: the (src, dst)
 * pair is written to cow (2 * max_pairs entries) and *n_cow counts the pairs (at
 * most one per call).  tokens (nullable) are the token ids; when given, blocks that
 * become full are registered in the prefix cache.  Returns PA_ERR_NO_SPACE, with
 * nothing changed, if the pool cannot hold the new blocks.
 */
pa_status pa_bm_append(pa_block_manager *bm, int64_t seq_id, const int32_t *tokens, int n,
                       int64_t *slots, int64_t *cow, int max_pairs, int *n_cow);

/* child (new id) shares all of parent's blocks: branching / beam search. */
pa_status pa_bm_fork(pa_block_manager *bm, int64_t parent_id, int64_t child_id);

/* End or cancel a sequence: its blocks are released at once. */
pa_status pa_bm_free(pa_block_manager *bm, int64_t seq_id);

/* Copy the block table (capacity entries at most) and lengths of a sequence. */
pa_status pa_bm_block_table(const pa_block_manager *bm, int64_t seq_id, int32_t *table,
                            int capacity, int *n_blocks, int64_t *context_len);

pa_status pa_bm_get_stats(const pa_block_manager *bm, pa_bm_stats *out);

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCKS_H */
