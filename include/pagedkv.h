/*
 * pagedkv.h -- C ABI of libpagedkv.so, the GB300 (sm_103a) paged KV-cache hot
 * path: page write (bf16 and int8), explicit gather, in-place paged decode
 * attention with split-KV, and chunked paged prefill attention.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every pointer argument is a caller-owned DEVICE pointer (allocated by the
 *    caller, e.g. through PyTorch) unless stated otherwise, 16-byte aligned.
 *    The calls of this header never allocate, free or synchronise; work is
 *    enqueued on `stream` (the last argument; NULL = the legacy default
 *    stream) and the call returns as soon as it is enqueued.  (The host-side
 *    block manager of pagedkv_blocks.h and the scratch pool of
 *    pagedkv_stream.h own host memory, and the latter a copy stream and
 *    events; their headers say so.)
 *  - Every call returns a PKV_* status.  Host-checkable argument errors are
 *    reported before anything is enqueued.  Errors that depend on device data
 *    (a table id outside [0, n_blocks], a position outside the table, a
 *    length too long) are found by the kernels, which skip the offending row
 *    and OR a PKV_DEV_* bit into *dev_status (a device int32; nullable: then
 *    the row is still skipped but nothing is reported).  No kernel traps.
 *  - No exception crosses the ABI.  Calls are thread-safe; calls enqueued on
 *    different streams that write the same memory race, as any CUDA work.
 *
 * Data layout (row-major, innermost last)
 * ---------------------------------------
 *  pool (per layer, K and V separately)  [n_blocks + 1][block_size][n_kv_heads][head_dim]
 *      bf16, or int8 codes with fp32 scales [n_blocks + 1][block_size][n_kv_heads].
 *      Row n_blocks is the scratch block: never allocated, the table entry of
 *      every unused logical block, and the target of writes from inactive
 *      sequences (tiny-llm paged_kv.py, PagedKVCache.__init__: "free slots
 *      write here").  Its contents are never read as data.
 *  block tables  int32 [n_seqs][max_blocks]; entry j = physical block of
 *      logical block j.  Token t of a sequence lives at pool row
 *      table[t / block_size] * block_size + t % block_size (tiny-llm
 *      paged_kv.py, module docstring; AstrAI cache.py, PagedCache.write).
 *      Entries at logical blocks >= ceil(len / block_size) are never read.
 *
 * Supported geometry: head_dim in {64, 128}; block_size a multiple of 16, at
 * most 256; n_q_heads % n_kv_heads == 0 and G = n_q_heads / n_kv_heads in
 * {1, 2, 4, 8} for decode (1 .. 16 dividing 64 for prefill); decode over int8
 * pages also needs n_kv_heads % 4 == 0 (else PKV_ERR_UNSUPPORTED); query head h
 * reads kv head h / G.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t pkv_bf16;                 /* raw bfloat16 bit pattern */
typedef struct CUstream_st *pkv_stream_t;  /* identical to cudaStream_t */

/* Return status of every call. */
enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, non-positive size, Hq % Hkv != 0 */
    PKV_ERR_UNSUPPORTED = 2,  /* head_dim, block_size, group size or kv dtype not supported */
    PKV_ERR_OUT_OF_RANGE = 3, /* a host-checkable size is out of range (e.g. n_new > table) */
    PKV_ERR_WORKSPACE = 4,    /* workspace null, smaller than required or not 256-byte aligned */
    PKV_ERR_CUDA = 5,         /* a CUDA call failed; pkv_last_cuda_error() says which */
    PKV_ERR_OUT_OF_BLOCKS = 6, /* block manager: not enough free blocks (nothing changed) */
    PKV_ERR_STATE = 7         /* block manager: the call does not fit the current state */
};

/* Bits OR-ed into *dev_status by the kernels. */
enum pkv_dev_status {
    PKV_DEV_BAD_BLOCK_ID = 1,        /* a table entry outside [0, n_blocks] was needed */
    PKV_DEV_BAD_POSITION = 2,        /* a write position < 0 or beyond the table width */
    PKV_DEV_BAD_LENGTH = 4,          /* a length < 0 or > max_blocks * block_size */
    PKV_DEV_WORKSPACE_OVERFLOW = 8,  /* decode work list larger than the workspace holds */
    PKV_DEV_TIMEOUT = 16             /* a bounded pipeline wait ran out (never expected) */
};

/* KV page formats (libmir-metal paged/mod.rs, KvPageFormat). */
enum pkv_kv_dtype { PKV_KV_BF16 = 0, PKV_KV_INT8 = 1 };

/* Pool geometry.  n_blocks = physical blocks EXCLUDING the scratch block. */
typedef struct pkv_dims {
    int32_t n_blocks;
    int32_t block_size;
    int32_t n_kv_heads;
    int32_t head_dim;
} pkv_dims;

/* Human-readable name of a PKV_* status. */
const char *pkv_status_string(int status);

/* The cudaError_t of the most recent PKV_ERR_CUDA on the calling thread (0 if none). */
int pkv_last_cuda_error(void);

/*
 * pkv_set_pipeline_wait_ns -- the limit of the kernels' pipeline waits, for
 * every launch prepared after the call (process-wide; 0 restores the default
 * of 4 s).  A wait that runs out sets PKV_DEV_TIMEOUT in dev_status and its
 * CTA winds down: the copies and tensor-core operations it already issued
 * finish (those waits keep the default limit) before it releases shared
 * memory or TMEM, and the call's outputs are then undefined.  The failure
 * path of the pages' Result-returning calls (libmir-metal paged/mod.rs,
 * PagedStore::update and context return errors instead of aborting); a short
 * limit makes that path run on purpose, for tests.  Returns the previous
 * limit.
 */
uint64_t pkv_set_pipeline_wait_ns(uint64_t ns);

/*
 * paged_kv_write -- native bf16 page write (tiny-llm paged_kv.py,
 * PagedLayerKV.update; AstrAI cache.py, PagedCache.write; libmir-metal
 * paged/mod.rs, write::native).
 *   k_new, v_new  bf16 [n_seqs][n_new][n_kv_heads][head_dim]   (read)
 *   k_pool,v_pool bf16 pools                                    (written)
 *   block_tables  int32 [n_seqs][max_blocks]; start_pos int32 [n_seqs]
 * For every s and j < n_new the K and V rows of token t = start_pos[s] + j are
 * copied bit-exactly to pool row table[s][t / bs] * bs + t % bs.  The caller
 * has already allocated the blocks.  A row whose block is outside the table
 * or names an id outside [0, n_blocks] is skipped (PKV_DEV_BAD_POSITION /
 * PKV_DEV_BAD_BLOCK_ID).  n_seqs == 0 or n_new == 0 is a no-op.
 */
int paged_kv_write(const pkv_bf16 *k_new, const pkv_bf16 *v_new, pkv_bf16 *k_pool,
                   pkv_bf16 *v_pool, pkv_dims dims, const int32_t *block_tables,
                   int32_t max_blocks, const int32_t *start_pos, int32_t n_seqs, int32_t n_new,
                   int32_t *dev_status, pkv_stream_t stream);

/*
 * paged_kv_write_int8 -- quantised page write (libmir-metal paged/mod.rs,
 * KvPageFormat::Int8PerTokenHead, write::quantized).  Same placement as
 * paged_kv_write; for each (token, kv head) row x of K and of V, in IEEE
 * binary32 with round-to-nearest-even:
 *   amax = max_d |x_d|;  scale = amax / 127;  code_d = clamp(rint(x_d / scale), -127, 127)
 * (a row of zeros stores scale 0 and codes 0).  Codes go to the int8 pools,
 * the scale to k_scales / v_scales [n_blocks + 1][block_size][n_kv_heads].
 */
int paged_kv_write_int8(const pkv_bf16 *k_new, const pkv_bf16 *v_new, int8_t *k_pool,
                        int8_t *v_pool, float *k_scales, float *v_scales, pkv_dims dims,
                        const int32_t *block_tables, int32_t max_blocks,
                        const int32_t *start_pos, int32_t n_seqs, int32_t n_new,
                        int32_t *dev_status, pkv_stream_t stream);

/*
 * paged_kv_gather -- explicit copy of each sequence's pages into a contiguous
 * view (tiny-llm paged_kv.py, PagedLayerKV.update gather -> (S, H, nb*bs, D);
 * AstrAI cache.py, PagedCache.gather; libmir-metal paged/mod.rs, context).
 *   k_out, v_out bf16 [n_seqs][n_kv_heads][out_tokens][head_dim]  (written)
 *   lens int32 [n_seqs]
 *   out[s][h][t][:] = pool[row of token t][h][:]  for t < lens[s];  0 for t >= lens[s].
 * bf16 pools only: quantised pages are consumed in place by
 * paged_decode_attention (libmir-metal refuses to gather them).  A length
 * outside [0, min(out_tokens, max_blocks * bs)] gives PKV_DEV_BAD_LENGTH and
 * that sequence's view is zero-filled.
 */
int paged_kv_gather(const pkv_bf16 *k_pool, const pkv_bf16 *v_pool, pkv_dims dims,
                    const int32_t *block_tables, int32_t max_blocks, const int32_t *lens,
                    int32_t n_seqs, int32_t out_tokens, pkv_bf16 *k_out, pkv_bf16 *v_out,
                    int32_t *dev_status, pkv_stream_t stream);

/*
 * paged_kv_copy_blocks -- copy whole pool blocks on the device: the device half
 * of copy-on-write for blocks shared between sequences (libmir-metal
 * paged/mod.rs, PagedStore::snapshot shares a sequence's pages by reference
 * count; a page that is still shared gets a private copy before it is written
 * -- pkv_bm_begin_step in pagedkv_blocks.h reports the pairs).
 *   pairs    int32 [n_pairs][2] device, 8-byte aligned: (source, destination)
 *            block ids in [0, n_blocks]
 *   k_pool, v_pool  bf16 pools (PKV_KV_BF16) or int8 code pools (PKV_KV_INT8,
 *            then k_scales / v_scales [n_blocks + 1][block_size][n_kv_heads]
 *            are copied too, else ignored)
 * For every pair, block destination becomes a bit-exact copy of block source
 * (all block_size rows, every kv head, K and V).  Destinations must be
 * distinct and no destination may be a source in the same call (the order of
 * the copies is not defined).  A pair naming an id outside [0, n_blocks] is
 * skipped (PKV_DEV_BAD_BLOCK_ID).  n_pairs == 0 is a no-op.
 */
int paged_kv_copy_blocks(const int32_t *pairs, int32_t n_pairs, void *k_pool, void *v_pool, float *k_scales,
                         float *v_scales, int32_t kv_dtype, pkv_dims dims, int32_t *dev_status,
                         pkv_stream_t stream);

/*
 * pkv_decode_workspace_bytes -- size of the workspace paged_decode_attention
 * needs (the per-store attention scratch of libmir-metal's
 * PagedAttentionScratch).  max_total_ctx_tokens bounds sum_s ctx_lens[s];
 * split_tokens as passed to paged_decode_attention (0 = automatic: the size
 * then covers every split the automatic choice can make).  Returns 0 on
 * invalid arguments, a max_total_ctx_tokens above n_seqs * INT32_MAX among
 * them.
 */
size_t pkv_decode_workspace_bytes(int32_t n_seqs, int32_t n_q_heads, int32_t head_dim,
                                  int64_t max_total_ctx_tokens, int32_t split_tokens);

/*
 * paged_decode_attention -- in-place paged GQA decode attention with split-KV
 * and a log-sum-exp merge (tiny-llm paged_kv.py docstring: the blocks are read
 * in place instead of gathered; metrale high_speed_swap impl_more.rs,
 * attend_layer_on_stream_with_q_pos: tiles with an online softmax joined by
 * one finalize).
 *   q        bf16 [n_seqs][n_q_heads][head_dim]
 *   k_pool, v_pool  bf16 pools (kv_dtype PKV_KV_BF16) or int8 code pools
 *            (PKV_KV_INT8, then k_scales / v_scales are required, else ignored)
 *   ctx_lens int32 [n_seqs]: tokens attended, INCLUDING the one just written
 *            (the decode mask k_pos <= len of tiny-llm's begin_step)
 *   out      bf16 [n_seqs][n_q_heads][head_dim]
 *   lse_out  fp32 [n_seqs][n_q_heads] natural-log log-sum-exp of the scaled
 *            scores (nullable)
 * For every sequence s and query head h (kv head g = h / G):
 *   o = softmax(softmax_scale * q K^T) V over the ctx_lens[s] tokens of s.
 * softmax_scale must be finite and positive (1/sqrt(head_dim) in the pages);
 * anything else returns PKV_ERR_INVALID_ARG.
 * The context is cut into logical ranges of split_tokens tokens (a multiple
 * of 16; 0 = automatic), each range is reduced with an online softmax, and
 * the ranges are merged by their log-sum-exp.  ctx_lens[s] == 0 gives o = 0
 * and lse = -inf.  workspace: device memory of at least
 * pkv_decode_workspace_bytes(...) bytes, 256-byte aligned (else
 * PKV_ERR_WORKSPACE; the CUDA allocators return such addresses), contents need
 * not be initialised, and it must not be shared by concurrently running calls.
 * With split_tokens = 0 and bf16 pages, a batch of at most one (sequence,
 * kv head) pair per SM whose table spans at most 256 tokens (head_dim 128) or
 * 512 (head_dim 64) is attended whole by one CTA per pair in a single launch
 * (same results within the tolerances; PKV_DECODE_IMPL=split in the
 * environment keeps the split-KV path).  PKV_DECODE_IMPL=tc runs int8 pages of
 * head_dim 128 with at most 8 query heads per kv head (n_kv_heads a multiple
 * of 4) on the tcgen05 tensor-core kernel instead of the mma.sync one (same
 * results within the int8 tolerance; slower on GB300 today).  The variable is
 * read at every call.
 */
int paged_decode_attention(const pkv_bf16 *q, int32_t n_q_heads, const void *k_pool,
                           const void *v_pool, const float *k_scales, const float *v_scales,
                           int32_t kv_dtype, pkv_dims dims, const int32_t *block_tables,
                           int32_t max_blocks, const int32_t *ctx_lens, int32_t n_seqs,
                           float softmax_scale, int32_t split_tokens, pkv_bf16 *out,
                           float *lse_out, void *workspace, size_t workspace_bytes,
                           int32_t *dev_status, pkv_stream_t stream);

/*
 * paged_decode_step -- one decode step of one layer in one call: the page
 * write of this step's new rows (paged_kv_write, or paged_kv_write_int8 when
 * kv_dtype is PKV_KV_INT8, with k_new / v_new / start_pos / n_new as there)
 * followed by paged_decode_attention over ctx_lens tokens, which must count
 * the rows just written.  Results are those of the two calls in sequence; the
 * write runs inside the first kernel launch of the decode, saving one launch
 * per layer (the per-layer step of tiny-llm paged_kv.py, PagedLayerKV.update:
 * write, then attention).
 */
int paged_decode_step(const pkv_bf16 *k_new, const pkv_bf16 *v_new, const int32_t *start_pos,
                      int32_t n_new, const pkv_bf16 *q, int32_t n_q_heads, void *k_pool,
                      void *v_pool, float *k_scales, float *v_scales, int32_t kv_dtype,
                      pkv_dims dims, const int32_t *block_tables, int32_t max_blocks,
                      const int32_t *ctx_lens, int32_t n_seqs, float softmax_scale,
                      int32_t split_tokens, pkv_bf16 *out, float *lse_out, void *workspace,
                      size_t workspace_bytes, int32_t *dev_status, pkv_stream_t stream);

/*
 * paged_prefill_attention -- chunked paged prefill (AstrAI cache.py,
 * PagedCache.write with seq_len > 1 followed by attention over the pages;
 * metrale impl_more.rs: a query at q_pos sees only slots <= q_pos of its last
 * block).  The chunk's K/V rows must already be in the pool (paged_kv_write
 * at start_pos = prefix_lens[s]).
 *   q, out   bf16 [n_seqs][chunk][n_q_heads][head_dim]
 *   lse_out  fp32 [n_seqs][chunk][n_q_heads] (nullable)
 *   prefix_lens int32 [n_seqs]
 * Query i of sequence s sits at absolute position P = prefix_lens[s] + i and
 * attends keys 0 .. P: the whole resident prefix plus, causally, the chunk up
 * to itself.  softmax_scale: finite and positive, as for the decode.  Q K^T
 * and P V run on the tcgen05 tensor cores.
 */
int paged_prefill_attention(const pkv_bf16 *q, int32_t n_q_heads, const pkv_bf16 *k_pool,
                            const pkv_bf16 *v_pool, pkv_dims dims, const int32_t *block_tables,
                            int32_t max_blocks, const int32_t *prefix_lens, int32_t n_seqs,
                            int32_t chunk, float softmax_scale, pkv_bf16 *out, float *lse_out,
                            int32_t *dev_status, pkv_stream_t stream);

/*
 * paged_decode_attention_noalloc -- paged_decode_attention for callers that
 * cannot allocate device memory.  The pages have no counterpart: this entry
 * point exists only for callers such as a plugin whose host framework owns all
 * device memory, or a runtime with a fixed memory budget, which may not call
 * cudaMalloc (or anything that allocates) to obtain a decode workspace.
 *
 * Arguments and results are those of paged_decode_attention, except that no
 * workspace is passed: the split-KV scratch is a static device array of
 * PKV_NOALLOC_DECODE_SCRATCH_BYTES (16 MiB) inside the library, which every
 * GPU that loads the library holds until the process exits.  The call
 * allocates nothing and frees nothing.
 *   max_total_ctx_tokens  an upper bound on sum_s ctx_lens[s]; when the
 *       scratch this needs (pkv_decode_workspace_bytes(n_seqs, n_q_heads,
 *       head_dim, max_total_ctx_tokens, split_tokens)) exceeds the static
 *       array, the call returns PKV_ERR_WORKSPACE and enqueues nothing.
 * The first call on a device looks up the array's device address (one
 * cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  The address is kept for the life of the
 * process, so a cudaDeviceReset after the first call is not supported.  A
 * max_total_ctx_tokens above n_seqs * INT32_MAX is PKV_ERR_INVALID_ARG.  All calls share the one array and it keeps the
 * last call's contents (nothing in it needs to start at zero: each call
 * rewrites what it reads).  Calls whose work overlaps on the GPU -- on
 * different streams, or from different threads without ordering -- race on
 * the scratch and give wrong results; order them on one stream.
 */
#define PKV_NOALLOC_DECODE_SCRATCH_BYTES (16u * 1024u * 1024u)

int paged_decode_attention_noalloc(const pkv_bf16 *q, int32_t n_q_heads, const void *k_pool,
                                   const void *v_pool, const float *k_scales,
                                   const float *v_scales, int32_t kv_dtype, pkv_dims dims,
                                   const int32_t *block_tables, int32_t max_blocks,
                                   const int32_t *ctx_lens, int32_t n_seqs, float softmax_scale,
                                   int32_t split_tokens, int64_t max_total_ctx_tokens,
                                   pkv_bf16 *out, float *lse_out, int32_t *dev_status,
                                   pkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
