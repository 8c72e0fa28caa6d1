/*
 * pagedkv_blocks.h -- host-side block manager that produces the block tables
 * the kernels of pagedkv.h consume: a fixed pool of equal-size blocks, a free
 * list, per-block reference counts (shared prefixes, forked sequences),
 * copy-on-write, and the per-step admission / growth / preemption rules of a
 * continuous-batching engine.
 *
 * Sources of the rules (the four pages this library follows):
 *   - tiny-llm paged_kv.py, BlockAllocator: blocks handed out lowest id first
 *     from a free stack and reused last-freed-first; freeing a block that is
 *     not in use is an error; a peak of blocks in use is kept.
 *   - AstrAI cache.py, PagedCache.alloc / alloc_n / free: a reference count
 *     per block, set to 1 on allocation and dropped by free (the block is free
 *     again at 0); a multi-block allocation is all or nothing.
 *   - libmir-metal paged/mod.rs, PagedStore::snapshot / release: a snapshot
 *     shares every page of a sequence by incrementing its reference count;
 *     release decrements them.
 *   - tiny-llm paged_kv.py, PagedKVCache.can_admit / admit / release /
 *     reserve_step / begin_step / end_step: admission needs ceil((n + 1) /
 *     block_size) free blocks per prompt (its blocks plus room for the first
 *     decode token); admit allocates ceil(n / block_size) blocks; before each
 *     decode step the newest sequences are preempted (their blocks freed) until
 *     every sequence that needs a new block can get one; begin_step gives each
 *     sequence whose blocks are full one more block; end_step counts the token.
 * Copy-on-write (a reading: the pages share pages but never write into a shared
 * one): when the block a sequence is about to write into is shared (reference
 * count > 1), begin_step gives the sequence a private copy -- a new block, the
 * old one's reference dropped -- and reports the (source, destination) pair,
 * which the caller copies on the device with paged_kv_copy_blocks before the
 * step's write.  reserve_step counts such copies as blocks needed.
 *
 * Conventions: host memory only, no CUDA calls; a manager is not thread-safe
 * (one thread, or the caller's lock, per manager).  Block ids are 0 ..
 * n_blocks - 1; the scratch id n_blocks marks unused table entries, as in the
 * kernels.  Every call returns a pkv_status; a failing call changes nothing.
 */
#ifndef PAGEDKV_BLOCKS_H
#define PAGEDKV_BLOCKS_H

#include "pagedkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_block_manager pkv_block_manager;

/*
 * pkv_bm_create -- n_blocks blocks of block_size tokens, n_slots sequence
 * slots, tables of max_blocks entries (a sequence holds at most
 * max_blocks * block_size tokens).  *out receives the manager (free it with
 * pkv_bm_destroy).  PKV_ERR_INVALID_ARG for non-positive sizes or a null out.
 */
int pkv_bm_create(int32_t n_blocks, int32_t block_size, int32_t n_slots, int32_t max_blocks,
                  pkv_block_manager **out);
void pkv_bm_destroy(pkv_block_manager *bm);

/* Block level (BlockAllocator / PagedCache.alloc, free). */
/* One block, lowest id first, last freed first; reference count 1. */
int pkv_bm_alloc(pkv_block_manager *bm, int32_t *block);
/* Drop one reference of each listed block; a block whose count reaches 0 goes
 * back on the free stack (in list order).  PKV_ERR_STATE if any block is not in
 * use (more references dropped than held), PKV_ERR_INVALID_ARG for a bad id. */
int pkv_bm_free(pkv_block_manager *bm, const int32_t *blocks, int32_t n);
int32_t pkv_bm_num_free(const pkv_block_manager *bm);
int32_t pkv_bm_peak_used(const pkv_block_manager *bm);
/* Reference count of a block (0 = free), -1 for an id outside [0, n_blocks). */
int32_t pkv_bm_refcount(const pkv_block_manager *bm, int32_t block);

/* Sequence slots (PagedKVCache scheduling, snapshot). */
/* *ok = 1 when sum over lengths of ceil((len + 1) / block_size) <= free blocks. */
int pkv_bm_can_admit(const pkv_block_manager *bm, const int32_t *lengths, int32_t n, int32_t *ok);
/* An inactive slot takes ceil(n_tokens / block_size) fresh blocks and holds
 * n_tokens tokens (all or nothing).  PKV_ERR_STATE if the slot is active,
 * PKV_ERR_OUT_OF_RANGE if n_tokens >= max_blocks * block_size. */
int pkv_bm_admit(pkv_block_manager *bm, int32_t slot, int32_t n_tokens);
/* Drop the slot's references and clear it (no-op for an inactive slot). */
int pkv_bm_release(pkv_block_manager *bm, int32_t slot);
/* An inactive dst shares every block of active src (references + 1) and holds
 * the same tokens; it is the newest admission. */
int pkv_bm_fork(pkv_block_manager *bm, int32_t src_slot, int32_t dst_slot);
/* Preempt the newest active sequences until the coming step's new blocks (full
 * tables plus copy-on-write) fit in the free ones; victims[] (n_slots entries)
 * receives the released slots, newest first, *n_victims their number. */
int pkv_bm_reserve_step(pkv_block_manager *bm, int32_t *victims, int32_t *n_victims);
/* Before the step's write at position len of every active slot: grow full
 * tables by one block, give shared write blocks a private copy.  copies
 * (2 * n_slots entries) receives (source, destination) pairs, *n_copies their
 * number.  PKV_ERR_OUT_OF_BLOCKS (nothing changed) when the free blocks do not
 * cover it -- call pkv_bm_reserve_step first; PKV_ERR_OUT_OF_RANGE if a
 * sequence is full. */
int pkv_bm_begin_step(pkv_block_manager *bm, int32_t *copies, int32_t *n_copies);
/* Every active slot now holds one more token. */
int pkv_bm_end_step(pkv_block_manager *bm);
/* Copy out the tables ([n_slots][max_blocks], unused entries = n_blocks),
 * token counts ([n_slots], 0 for inactive slots) and active flags ([n_slots]);
 * any of the three may be null. */
int pkv_bm_export(const pkv_block_manager *bm, int32_t *tables, int32_t *lens, int32_t *active);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_BLOCKS_H */
