/*
 * pagedkv_stream.h -- decode attention over more blocks than the device holds:
 * the blocks live in a host tier (pinned host memory, the pool layout of
 * pagedkv.h, bf16), a device scratch pool holds n_slots of them, and the decode
 * streams each sequence's blocks through the scratch pool one tile of at most
 * n_slots blocks at a time (metrale high_speed_swap impl_more.rs,
 * attend_layer_on_stream_with_q_pos: look up resident blocks, assign scratch
 * slots to the missing ones and read them from the tier, attend the tile with
 * the running softmax state -- step_tile -- and finalize after the last tile).
 * The block predictor of that page is not built: slots are reused least
 * recently used first.  A rewritten host block must be dropped from the
 * scratch pool (pkv_sp_invalidate), as the page's offload does.
 *
 * On GB300 the staging is one kernel that reads the host tier directly over the
 * CPU-GPU link (pinned host memory is mapped into the device address space);
 * the calls below check that mapping with cudaHostGetDevicePointer and return
 * PKV_ERR_INVALID_ARG for host buffers that are not pinned and mapped.
 */
#ifndef PAGEDKV_STREAM_H
#define PAGEDKV_STREAM_H

#include "pagedkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_scratch_pool pkv_scratch_pool;

/*
 * pkv_sp_create -- residency bookkeeping for a device scratch pool of n_slots
 * blocks (slot ids 0 .. n_slots - 1; the device pool tensors have n_slots + 1
 * blocks, the last a scratch block) and per-tile plans for batches of up to
 * max_seqs sequences.  Holds two small pinned host staging buffers (the plan of
 * a tile is copied to the device from them) and, from the first
 * paged_decode_streamed call on, a copy stream and events of the device that
 * was current then (the pool serves that device only).  Not thread-safe.
 */
int pkv_sp_create(int32_t n_slots, int32_t max_seqs, pkv_scratch_pool **out);
void pkv_sp_destroy(pkv_scratch_pool *sp);
/* Slot holding host block b, or -1 when it is not resident. */
int32_t pkv_sp_lookup(const pkv_scratch_pool *sp, int32_t host_block);
/* Forget the resident copy of host block b (after the tier copy was rewritten). */
int pkv_sp_invalidate(pkv_scratch_pool *sp, int32_t host_block);

/*
 * pkv_sp_plan_tile -- the plan of the next tile (host only; paged_decode_streamed
 * calls it per tile): starting at cursor[0] = sequence, cursor[1] = block of
 * that sequence, take the batch's blocks in order until tile_blocks blocks
 * (<= 0 or > n_slots: n_slots) or the end.  Each block reuses its resident
 * slot, or takes the least recently used slot not yet used by this tile (its
 * old block is forgotten) and adds (host block, slot) to pairs [n_slots][2]
 * (*n_pairs of them).  With tile_blocks <= n_slots / 2 a tile never stages
 * into a slot the tile before it uses (those are the most recently used).
 * tile_tables [n_seqs][W], W = min(tile cap, max_blocks), receives each
 * sequence's slots in token order (unused entries = n_slots, the scratch
 * slot), tile_lens [n_seqs] its tokens in this tile.  Advances cursor; *done =
 * 1 when no block is left.  A negative host id among the tile's blocks returns
 * PKV_ERR_OUT_OF_RANGE before any state changes.  The residency index takes
 * 4 bytes per host block up to the largest id seen.
 */
int pkv_sp_plan_tile(pkv_scratch_pool *sp, const int32_t *host_tables, int32_t max_blocks, const int32_t *ctx_lens,
                     int32_t n_seqs, int32_t block_size, int32_t tile_blocks, int32_t *cursor, int32_t *tile_tables,
                     int32_t *tile_lens, int32_t *pairs, int32_t *n_pairs, int32_t *done);

/*
 * paged_kv_stage_blocks -- copy host-tier blocks into scratch-pool slots on the
 * device: pairs int32 [n_pairs][2] device (host block in [0, n_host_blocks),
 * slot in [0, pool_dims.n_blocks]); host_k / host_v pinned host memory
 * [n_host_blocks][block_size][n_kv_heads][head_dim] bf16; pool_k / pool_v
 * device [pool_dims.n_blocks + 1][...] bf16.  Destination slots must be
 * distinct.  Out-of-range ids are skipped (PKV_DEV_BAD_BLOCK_ID).  Returns
 * PKV_ERR_INVALID_ARG for a negative count or size, a null or misaligned
 * pointer (pairs 8-byte, the rest 16-byte aligned) or host memory that is not
 * pinned and mapped; PKV_ERR_UNSUPPORTED for head_dim outside {64, 128}.
 */
int paged_kv_stage_blocks(const int32_t *pairs, int32_t n_pairs, const pkv_bf16 *host_k, const pkv_bf16 *host_v,
                          int32_t n_host_blocks, pkv_bf16 *pool_k, pkv_bf16 *pool_v, pkv_dims pool_dims,
                          int32_t *dev_status, pkv_stream_t stream);

/* Device workspace paged_decode_streamed needs (0 for invalid arguments). */
size_t pkv_streamed_workspace_bytes(int32_t n_seqs, int32_t n_q_heads, int32_t head_dim, int32_t n_slots,
                                    int32_t block_size);

/*
 * paged_decode_streamed -- o = softmax(softmax_scale * q K^T) V over the
 * ctx_lens[s] tokens of each sequence, whose blocks are host_tables[s][j]
 * (HOST int32 [n_seqs][max_blocks], ids into the host tier).  The tokens of
 * the batch are taken in order (sequence by sequence) in tiles of
 * n_slots = pool_dims.n_blocks blocks when the batch fits the scratch pool,
 * else of n_slots / 2 blocks; for each tile the resident blocks are reused,
 * the missing ones staged (paged_kv_stage_blocks, on the pool's copy stream,
 * overlapping the attention of the tile before), the tile attended by the
 * split-KV decode of pagedkv.h over the scratch pool, and its result merged
 * into a float32 running (output, log-sum-exp) state; the last step
 * writes out (bf16 [n_seqs][n_q_heads][head_dim]) and lse_out (fp32
 * [n_seqs][n_q_heads], natural log; nullable).  ctx_lens is HOST int32
 * [n_seqs]; q, out, lse_out device.  workspace: device memory of
 * pkv_streamed_workspace_bytes(...) bytes, 256-byte aligned (else
 * PKV_ERR_WORKSPACE); the residency state in sp carries
 * over between calls (a later call reuses what is still resident).  The
 * attention and merges are enqueued on stream, the plan copies and staging on
 * the pool's copy stream, ordered against stream by events (the staging waits
 * for the work enqueued on stream before the call; the result is complete
 * when stream reaches the end of the call).  The call returns once every tile
 * is enqueued (it waits on the host only until the plan of the tile two
 * before has been copied).  The scratch pool and workspace must not be used by
 * other work meanwhile.  An error return after the first tile was planned
 * (PKV_ERR_CUDA) leaves the residency bookkeeping ahead of what reached the
 * device: destroy the scratch pool (or invalidate every block) before
 * reusing it.
 */
int paged_decode_streamed(const pkv_bf16 *q, int32_t n_q_heads, const pkv_bf16 *host_k, const pkv_bf16 *host_v,
                          int32_t n_host_blocks, pkv_bf16 *pool_k, pkv_bf16 *pool_v, pkv_dims pool_dims,
                          pkv_scratch_pool *sp, const int32_t *host_tables, int32_t max_blocks,
                          const int32_t *ctx_lens, int32_t n_seqs, float softmax_scale, pkv_bf16 *out,
                          float *lse_out, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                          pkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_STREAM_H */
