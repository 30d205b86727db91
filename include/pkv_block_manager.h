/*
 * pkv_block_manager.h -- C ABI of the host-side block manager of libpkv:
 * the bookkeeping that feeds the paged KV cache's write and decode calls
 * (pkv.h) with slot mappings, block tables and context lengths.
 *
 * What it manages, as the pages describe it:
 *   - The KV cache is a pool of fixed-size physical blocks; a sequence grows
 *     one block at a time and its blocks live anywhere in the pool; a block
 *     table maps logical block index -> physical block, and slot_mapping is
 *     the write-side view (token -> flat physical slot block * bs + offset).
 *     Interview note "PagedAttention kernel: paged KV cache 与 block table",
 *     section 直接答案 and follow-up questions 面试官追问 (growth = allocate a
 *     page; sharing = two tables pointing at one physical block).
 *   - Prefix caching: sequences whose prompts share a prefix point their
 *     tables at the same physical blocks for that prefix; the block is the
 *     unit of sharing (same note, 面试官追问 on prefix caching).
 *   - The blog post on re-implementing paged attention (jsqmd.com, news
 *     887134): a block manager with a free-block queue, a set of used blocks,
 *     a map from a block's hash -- computed from its token ids and the hash
 *     of the prefix before it -- to the block holding them, an allocate call
 *     that returns how much of the prompt is already cached, and an LRU
 *     policy for cached blocks left as future work.
 *
 * Design (this library's reading):
 *   - Only FULL blocks are hashed and shared.  A full block is registered
 *     under hash(parent hash, its bs token ids) and remembers its parent
 *     block and token ids; a lookup matches only if the parent block and
 *     every token id are equal, so a hash collision can never share wrong
 *     data.  A sequence's last, partly filled block is always its own, so
 *     appends never write into a shared block (no copy-on-write needed).
 *   - Reference counts: a block is owned by every sequence whose table holds
 *     it.  When the count drops to zero the block goes to the free list; a
 *     registered block keeps its contents and registration there and can be
 *     revived by a later prefix match.  Allocation takes unregistered free
 *     blocks first, then registered ones least recently freed first (LRU),
 *     dropping their registration.
 *   - Every call either succeeds completely or changes nothing (a request
 *     that needs more free blocks than there are returns
 *     PKV_ERR_OUT_OF_BLOCKS with the state unchanged).
 *   - Host memory only; no CUDA call.  A handle may be used from several
 *     threads: calls on one handle are serialised by an internal lock.
 *
 * Ownership: the manager owns its handle (pkv_bm_destroy frees it); every
 * array argument is caller-owned host memory, read or written only during
 * the call.
 */
#ifndef PKV_BLOCK_MANAGER_H
#define PKV_BLOCK_MANAGER_H

#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_block_manager pkv_block_manager;

/*
 * pkv_bm_create -- a manager of num_blocks physical blocks of block_size
 * tokens (both > 0; num_blocks < 2^31).  prefix_caching != 0 enables the
 * sharing of full prompt blocks.  *out receives the handle.
 * Errors: PKV_ERR_INVALID_ARG for bad sizes or a NULL out.
 */
PKV_API pkv_status pkv_bm_create(int64_t num_blocks, int block_size, int prefix_caching,
                                 pkv_block_manager **out);

/* pkv_bm_destroy -- frees the handle (NULL is a no-op). */
PKV_API void pkv_bm_destroy(pkv_block_manager *bm);

/*
 * pkv_bm_add_sequence -- admit sequence seq_id (>= 0, not already live)
 * with its prompt token_ids[0 .. ntoken) (ntoken >= 1).  Its blocks are
 * allocated; with prefix caching the longest run of leading full blocks
 * already cached is shared instead.
 *   slot_mapping  [ntoken] out (may be NULL): the slot of every prompt
 *                 token whose K/V the caller must write, -1 for tokens
 *                 already cached -- ready for pkv_write, which skips
 *                 negative slots.
 *   num_cached    out (may be NULL): how many leading prompt tokens are
 *                 cached (a multiple of block_size).
 * The prompt's full blocks are registered at once: a sequence admitted
 * after this call may share them (its slots for them come back -1), so the
 * caller writes every returned slot before any attention reads either.
 * Errors: PKV_ERR_INVALID_ARG (bad id, duplicate id, bad arguments),
 * PKV_ERR_OUT_OF_BLOCKS.
 */
PKV_API pkv_status pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq_id,
                                       const int64_t *token_ids, int64_t ntoken,
                                       int64_t *slot_mapping, int64_t *num_cached);

/*
 * pkv_bm_append_tokens -- one decode step: for i in [0, B), append token
 * token_ids[i] to live sequence seq_ids[i] and return its slot in
 * slot_mapping[i]; a negative seq_ids[i] is a padding entry and gets slot
 * -1.  A sequence crossing a block edge gets a new block; a block that
 * fills up is registered for prefix sharing.  Each live id at most once.
 * Errors: PKV_ERR_INVALID_ARG (unknown or repeated id),
 * PKV_ERR_OUT_OF_BLOCKS (nothing appended).
 */
PKV_API pkv_status pkv_bm_append_tokens(pkv_block_manager *bm, const int64_t *seq_ids,
                                        const int64_t *token_ids, int B, int64_t *slot_mapping);

/*
 * pkv_bm_free_sequence -- release a live sequence's blocks (their counts
 * drop; blocks that reach zero go to the free list, registered ones kept
 * for reuse until evicted).  Errors: PKV_ERR_INVALID_ARG (unknown id).
 */
PKV_API pkv_status pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq_id);

/*
 * pkv_bm_build_batch -- the decode batch for B entries: row i of
 * block_tables [B, max_blocks] int32 is the table of live sequence
 * seq_ids[i] followed by `tail` in every unused entry, context_lens[i] its
 * length; a negative seq_ids[i] is padding (length 0, whole row `tail`).
 * Errors: PKV_ERR_INVALID_ARG (unknown id, a table longer than max_blocks,
 * bad arguments).
 */
PKV_API pkv_status pkv_bm_build_batch(pkv_block_manager *bm, const int64_t *seq_ids, int B,
                                      int max_blocks, int32_t tail, int32_t *block_tables,
                                      int32_t *context_lens);

/*
 * pkv_bm_sequence_info -- length and table of a live sequence:
 * *context_len tokens in *num_table_blocks blocks; the first
 * min(*num_table_blocks, max_blocks) entries are written to table (may be
 * NULL with max_blocks 0).  Errors: PKV_ERR_INVALID_ARG (unknown id).
 */
PKV_API pkv_status pkv_bm_sequence_info(pkv_block_manager *bm, int64_t seq_id,
                                        int64_t *context_len, int *num_table_blocks,
                                        int32_t *table, int max_blocks);

/*
 * pkv_bm_stats -- counts: free blocks (including cached ones with no
 * owner), blocks holding a registered full block, live sequences.  Any
 * pointer may be NULL.
 */
PKV_API void pkv_bm_stats(pkv_block_manager *bm, int64_t *free_blocks, int64_t *cached_blocks,
                          int64_t *live_sequences);

/*
 * pkv_bm_block_refcount -- owners of physical block `block` (0 when free),
 * or -1 for a block id outside the pool.
 */
PKV_API int pkv_bm_block_refcount(pkv_block_manager *bm, int64_t block);

#ifdef __cplusplus
}
#endif

#endif /* PKV_BLOCK_MANAGER_H */
