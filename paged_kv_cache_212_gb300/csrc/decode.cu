// decode.cu -- in-place paged GQA decode attention with split-KV and a
// log-sum-exp merge, for bf16 pages and for int8 pages with fp32 per-(token,
// kv head) scales.
//
// Three launches on the caller's stream, no host synchronisation:
//   1. decode_plan_kernel (one CTA) cuts the work into items.  With
//      split_tokens > 0 an item is one logical range [k S, (k+1) S) of one
//      sequence (metrale high_speed_swap impl_more.rs,
//      attend_layer_on_stream_with_q_pos: tiles of resident blocks).  With
//      split_tokens == 0 the concatenated 16-token stages of all sequences are
//      cut into equal contiguous ranges, about one per CTA, so every CTA gets
//      the same amount of work; a range may cover the end of one sequence and
//      the start of the next.  Each (sequence, item) piece owns one partial
//      slot.  The plan also resets the work counter.
//   2. decode_split_kernel (persistent, one or two CTAs per SM): lane 0 of a
//      producer warp takes (item, kv-head group) units (CTA b: units b,
//      b + grid, ... when the items are the equal balanced ones; the next from
//      the counter for fixed splits) and streams the item's pages, 16 tokens
//      per stage, into a shared-memory ring with TMA
//      (cp.async.bulk.tensor, 128-byte swizzle), addressed through the block
//      table.  One consumer warp per kv head contracts the stage with its GQA
//      query group on the tensor cores (mma.sync m16n8k16: S^T = K Q^T with the
//      16 tokens as M and the query heads as N, then O^T += V^T P^T) and keeps
//      an online softmax (running max and sum in log2 units).  A sequence in
//      one piece writes its output directly; otherwise each piece writes its
//      partial (m, l, acc) to the workspace.
//   3. decode_merge_kernel, for sequences in two or more pieces (a warp per
//      (sequence, query head) pair at a time):
//      o = sum_k 2^(m_k - M) acc_k / sum_k 2^(m_k - M) l_k (the finalize step
//      of the tiled attention) and lse = ln 2 (M + log2 L).
// The split and merge kernels are programmatic dependent launches: each
// starts while its predecessor drains and waits (griddepcontrol.wait) before
// reading the predecessor's results.
//
// Pool tiles in shared memory: for each stage and each 64-element half of
// head_dim, a [heads][16 tokens][128 bytes] box with the TMA 128-byte swizzle
// (16-byte chunk c of row r stored at chunk c ^ (r & 7)), so ldmatrix reads of
// eight consecutive tokens hit eight different bank groups.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"
#include "write_rows.cuh"

namespace pkv {

namespace {

constexpr int kStageTokens = 16;
constexpr int kMaxStages = 8;
// the running maximum of the online softmax lags the true one by at most this
// (log2 units): probabilities stay at most 2^8
constexpr float kLazyMax = 8.0f;
constexpr uint32_t kHdrCounter = 0, kHdrTotal = 1, kHdrOverflow = 2, kHdrChunk = 3, kHdrStages = 4;
constexpr int32_t kMinChunkStages = 4;   // balanced items hold at least 64 tokens

enum : int32_t { kMetaFirst = 1, kMetaLast = 2, kMetaBad = 4, kMetaStop = 8, kMetaFinal = 16, kMetaPad = 32 };

// L2 eviction priorities for the split-KV partials: the split kernel stores
// them to be evicted last, so that they are still in L2 when the merge reads
// them after the whole context has streamed through; the merge's reads mark
// them to be evicted first (they are dead until the next call writes them).
__device__ __forceinline__ uint64_t l2_evict_last_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void st_kept(float *a, float v, uint64_t pol)
{
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(a), "f"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_kept(float2 *a, float2 v, uint64_t pol)
{
    asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;" ::"l"(a), "f"(v.x), "f"(v.y), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ float2 ld_last_use(const float2 *a, uint64_t pol)
{
    float2 v;
    asm volatile("ld.global.cg.L2::cache_hint.v2.f32 {%0, %1}, [%2], %3;" : "=f"(v.x), "=f"(v.y) : "l"(a), "l"(pol));
    return v;
}
// drops a 128-byte L2 line without writing it back (its contents become
// undefined): partial rows the merge has read are dead until the next call
__device__ __forceinline__ void l2_discard_line(const void *a)
{
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(a) : "memory");
}
__device__ __forceinline__ float4 ld_last_use(const float4 *a, uint64_t pol)
{
    float4 v;
    asm volatile("ld.global.cg.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(a), "l"(pol));
    return v;
}

struct StageMeta {
    int32_t seq;
    int32_t split_index;  // the piece's partial slot
    int32_t n_valid;      // valid tokens in this stage (1..16)
    int32_t flags;
    int32_t head_group;   // which group of hpc kv heads the item covers
    int32_t n_splits;     // pieces of this sequence
    int32_t row0;         // pool row of the stage's first token (when its block is valid)
    int32_t pad;
};

struct DecodeParams {
    const __nv_bfloat16 *q;
    int32_t n_q_heads, group, hpc, n_hg;
    int32_t n_blocks, block_size, n_kv_heads;
    const int32_t *tables;
    int32_t max_blocks;
    const int32_t *ctx_lens;
    int32_t n_seqs;
    float scale_log2;
    int32_t split_tokens;         // 0: balanced pieces
    __nv_bfloat16 *out;
    float *lse_out;
    DecodeWorkspace ws;
    int32_t *dev_status;
    int32_t n_stages;
    int32_t boxes_per_half;  // TMA boxes per (K or V, half): 1 (all heads) or hpc (one per head)
    uint32_t stage_bytes, tx_bytes, kv_tile_bytes, scale_tile_bytes, q_slot_bytes;
    int32_t scale_heads;          // int8: kv heads per scale box (a multiple of 4: 16-byte rows)
    int32_t scales_in_stage;      // int8: 1 = the scale rows come with each stage (TMA), 0 = the
                                  // consumers read them from k_scales / v_scales themselves
    const float *k_scales, *v_scales;
    int32_t tile_stages;          // > 1: each piece is padded to a multiple of this many stages
    unsigned long long wait_ns;   // limit of the pipeline waits
};

// Shared-memory carve-up (dynamic smem, base rounded up to 1024 bytes).
struct SmemLayout {
    uint8_t *stages;     // n_stages * stage_bytes
    uint8_t *q_slots;    // 2 * q_slot_bytes
    uint64_t *full_bar, *empty_bar, *qfull_bar, *qempty_bar;
    StageMeta *meta;
    int32_t *abort_flag;
};

__device__ __forceinline__ SmemLayout carve(uint8_t *smem, const DecodeParams &p)
{
    SmemLayout L;
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem) + 1023) &
                                                ~uintptr_t(1023));
    L.stages = base;
    base += (size_t)p.n_stages * p.stage_bytes;
    L.q_slots = base;
    base += 2 * (size_t)p.q_slot_bytes;
    L.full_bar = reinterpret_cast<uint64_t *>(base);
    L.empty_bar = L.full_bar + kMaxStages;
    L.qfull_bar = L.empty_bar + kMaxStages;
    L.qempty_bar = L.qfull_bar + 2;
    L.meta = reinterpret_cast<StageMeta *>(L.qempty_bar + 2);
    L.abort_flag = reinterpret_cast<int32_t *>(L.meta + kMaxStages);
    return L;
}

__host__ __device__ constexpr size_t smem_tail_bytes()
{
    return (2 * kMaxStages + 4) * sizeof(uint64_t) + kMaxStages * sizeof(StageMeta) + 16;
}

// int8 -> fp16 for four packed codes with a bias: (0x6400 | (b ^ 0x80)) is
// the fp16 value 1152 + b, exact for every code b.  Products of the biased
// codes are corrected once per score (S - 1152 sum_d q_d) and once per output
// (O - 1152 sum_t p_t) instead of subtracting the bias from every element.
constexpr float kCodeBias = 1152.0f;
__device__ __forceinline__ void int8x4_to_biased_half2x2(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    const uint32_t u = w ^ 0x80808080u;
    lo = __byte_perm(u, 0x64646464u, 0x4140);
    hi = __byte_perm(u, 0x64646464u, 0x4342);
}

// Byte offset of the 16-byte chunk `chunk` (0..7) of row `row` in a
// 128-byte-swizzled tile of 128-byte rows.
__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk)
{
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

}  // namespace

// ---------------------------------------------------------------------------
// 1. plan
// ---------------------------------------------------------------------------

// Exclusive prefix sum of v over the CTA (blockDim.x a multiple of 32);
// *total receives the CTA-wide sum.  scratch: 33 ints of shared memory.
__device__ int32_t block_exclusive_scan(int32_t v, int32_t *total, int32_t *scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t u = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += u;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int32_t x = lane < (int)(blockDim.x >> 5) ? scratch[lane] : 0;
        int32_t xi = x;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t u = __shfl_up_sync(0xffffffffu, xi, off);
            if (lane >= off) xi += u;
        }
        scratch[lane] = xi - x;
        if (lane == 31) scratch[32] = xi;
    }
    __syncthreads();
    const int32_t r = scratch[warp] + incl - v;
    *total = scratch[32];
    __syncthreads();
    return r;
}

// Inclusive warp scan.
__device__ __forceinline__ int32_t warp_inclusive_scan(int32_t v, int lane)
{
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t u = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += u;
    }
    return v;
}

// The plan of a batch of at most kSmallPlanSeqs sequences, made by one warp:
// lane l holds sequences 4l .. 4l + 3, and each pass is one warp scan (no
// block barrier, ctx_lens read once).  Same results as the block-wide plan.
constexpr int32_t kSmallPlanSeqs = 128;
__device__ void plan_small(const int32_t *__restrict__ ctx_lens, int32_t n_seqs, int32_t split_tokens,
                           int32_t max_tokens, int32_t n_q_heads, int32_t head_dim, int32_t items_target,
                           DecodeWorkspace ws, __nv_bfloat16 *out, float *lse_out, int32_t *dev_status)
{
    const int lane = threadIdx.x & 31;
    const bool balanced = split_tokens == 0;
    const int32_t unit = balanced ? kStageTokens : split_tokens;
    int32_t ctx[4], n[4], pre[4];
    int32_t loc = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int32_t sq = 4 * lane + j;
        ctx[j] = sq < n_seqs ? ctx_lens[sq] : -1;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int32_t sq = 4 * lane + j;
        n[j] = 0;
        if (sq < n_seqs) {
            if (ctx[j] < 0 || ctx[j] > max_tokens)
                report(dev_status, PKV_DEV_BAD_LENGTH);
            else
                n[j] = (ctx[j] + unit - 1) / unit;
        }
        loc += n[j];
    }
    const int32_t incl = warp_inclusive_scan(loc, lane);
    const int32_t total = __shfl_sync(0xffffffffu, incl, 31);
    int32_t ex = incl - loc;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        pre[j] = ex;
        ex += n[j];
    }
    int32_t n_items = 0, chunk = 0;
    bool overflow = false;
    if (!balanced) {
        n_items = total;
        overflow = total > ws.capacity;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int32_t sq = 4 * lane + j;
            if (sq >= n_seqs) continue;
            ws.seg[sq] = make_int2(pre[j], n[j]);
            for (int32_t k = 0; k < n[j]; ++k)
                if (pre[j] + k < ws.capacity) ws.items[pre[j] + k] = make_int2(sq, k);
        }
    } else {
        if (lane == 0) ws.seq_prefix[n_seqs] = total;
        const int32_t room = ws.capacity - n_seqs;
        overflow = room < 1 && total > 0;
        if (total > 0 && !overflow) {
            const int32_t want = max(1, min(items_target, room));
            chunk = max(kMinChunkStages, (total + want - 1) / want);
            n_items = (total + chunk - 1) / chunk;
        }
        int32_t np[4], loc2 = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            np[j] = chunk > 0 && n[j] > 0 ? (pre[j] + n[j] - 1) / chunk - pre[j] / chunk + 1 : 0;
            loc2 += np[j];
        }
        const int32_t incl2 = warp_inclusive_scan(loc2, lane);
        int32_t ex2 = incl2 - loc2;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int32_t sq = 4 * lane + j;
            if (sq < n_seqs) {
                ws.seq_prefix[sq] = pre[j];
                ws.seg[sq] = make_int2(ex2, np[j]);
                // items whose first stage lies in this sequence start with it
                // (none when the work list overflowed: chunk is then 0)
                for (int32_t i = (pre[j] + chunk - 1) / max(chunk, 1);
                     chunk > 0 && n[j] > 0 && i * chunk < pre[j] + n[j]; ++i)
                    ws.items[i] = make_int2(sq, 0);
            }
            ex2 += np[j];
        }
    }
    if (lane == 0) {
        if (overflow) report(dev_status, PKV_DEV_WORKSPACE_OVERFLOW);
        ws.header[kHdrTotal] = overflow ? 0u : (uint32_t)n_items;
        ws.header[kHdrOverflow] = overflow ? 1u : 0u;
        ws.header[kHdrChunk] = (uint32_t)chunk;
        ws.header[kHdrStages] = balanced && !overflow ? (uint32_t)total : 0u;
        ws.header[kHdrCounter] = 0u;
    }
    // sequences no piece will cover get o = 0 and lse = -inf
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int32_t sq = 4 * lane + j;
        if (sq >= n_seqs || (!overflow && ctx[j] > 0 && ctx[j] <= max_tokens)) continue;
        const int64_t row = (int64_t)sq * n_q_heads;
        uint4 *o = reinterpret_cast<uint4 *>(out + row * head_dim);
        for (int32_t i = 0; i < n_q_heads * head_dim / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
        if (lse_out)
            for (int32_t i = 0; i < n_q_heads; ++i) lse_out[row + i] = -INFINITY;
    }
}

// 256-thread CTAs for the plan launch: small enough to be placed on an SM
// beside the previous kernels' CTAs, so they are resident and waiting when
// their predecessor completes.
constexpr int kPlanThreads = 256;

// CTA 0 plans; in the fused decode step, CTAs 1.. also write this step's new
// K/V rows into the pool (write_mode 1: bf16 copy, 2: int8 quantisation), so
// the split kernel, which waits for this whole grid, reads them.
__global__ void __launch_bounds__(kPlanThreads, 4) decode_plan_kernel(const int32_t *__restrict__ ctx_lens,
                                                           int32_t n_seqs, int32_t split_tokens,
                                                           int32_t max_tokens, int32_t n_q_heads,
                                                           int32_t head_dim, int32_t n_kv_heads,
                                                           int32_t items_target, DecodeWorkspace ws,
                                                           __nv_bfloat16 *out, float *lse_out,
                                                           int32_t *dev_status, const WriteArgs w, int32_t write_mode,
                                                           float *k_scales, float *v_scales)
{
    __shared__ int32_t scratch[33];
    grid_dependents_launch();   // the split kernel may start; it waits for this grid's results
    grid_dependency_wait();     // launched as a dependent of the previous kernel: wait for its results
    if (blockIdx.x > 0) {
        const int64_t wb = blockIdx.x - 1, nwb = gridDim.x - 1;
        if (write_mode == 1) {
            write_bf16_vectors(w, wb * blockDim.x + threadIdx.x, nwb * blockDim.x);
        } else if (write_mode == 2) {
            const int64_t warps = blockDim.x >> 5;
            if (head_dim == 128)
                write_int8_units<16>(w, k_scales, v_scales, wb * warps + (threadIdx.x >> 5), nwb * warps);
            else
                write_int8_units<8>(w, k_scales, v_scales, wb * warps + (threadIdx.x >> 5), nwb * warps);
        }
        return;
    }
    if (n_seqs <= kSmallPlanSeqs) {
        if (threadIdx.x < 32)
            plan_small(ctx_lens, n_seqs, split_tokens, max_tokens, n_q_heads, head_dim, items_target, ws, out,
                       lse_out, dev_status);
        return;
    }
    const int tid = threadIdx.x;
    const bool balanced = split_tokens == 0;
    const int32_t unit = balanced ? kStageTokens : split_tokens;
    // Each thread keeps the lengths and prefixes of its first kCache sequences
    // (s = tid + c * blockDim.x) in registers across the passes, so a batch of
    // up to kCache * blockDim.x sequences reads ctx_lens once and never reads
    // back what the plan wrote; larger batches re-read the rest.
    constexpr int kCache = 4;
    int32_t ctx_c[kCache] = {}, ex_c[kCache] = {};
    auto ctx_of = [&](int c, int32_t s) { return c < kCache ? ctx_c[c] : (s < n_seqs ? ctx_lens[s] : -1); };
    // pass 1: units (16-token stages, or fixed splits) per sequence and their prefix
    int32_t running = 0;
#pragma unroll
    for (int c = 0; c < kCache + 1; ++c) {
        for (int32_t c0 = c * (int32_t)blockDim.x; c0 < n_seqs; c0 += (c < kCache ? n_seqs : (int32_t)blockDim.x)) {
            const int32_t s = c0 + tid;
            const int32_t ctx = s < n_seqs ? ctx_lens[s] : -1;
            int32_t n = 0;
            if (s < n_seqs) {
                if (ctx < 0 || ctx > max_tokens)
                    report(dev_status, PKV_DEV_BAD_LENGTH);
                else
                    n = (ctx + unit - 1) / unit;
            }
            int32_t tot;
            const int32_t ex = running + block_exclusive_scan(n, &tot, scratch);
            if (c < kCache) {
                ctx_c[c] = ctx;
                ex_c[c] = ex;
            }
            if (s < n_seqs) {
                if (balanced) {
                    ws.seq_prefix[s] = ex;
                } else {
                    ws.seg[s] = make_int2(ex, n);
                    for (int32_t k = 0; k < n; ++k)
                        if (ex + k < ws.capacity) ws.items[ex + k] = make_int2(s, k);
                }
            }
            running += tot;
        }
    }
    int32_t n_items = 0, chunk = 0;
    const int32_t total_stages = running;
    bool overflow = false;
    if (!balanced) {
        n_items = running;
        overflow = running > ws.capacity;
    } else {
        const int32_t total = running;
        if (tid == 0) ws.seq_prefix[n_seqs] = total;
        const int32_t room = ws.capacity - n_seqs;   // items the partial slots allow
        overflow = room < 1 && total > 0;
        if (total > 0 && !overflow) {
            const int32_t want = max(1, min(items_target, room));
            chunk = max(kMinChunkStages, (total + want - 1) / want);
            n_items = (total + chunk - 1) / chunk;
        }
        // pass 2: pieces per sequence, their slots, and the first sequence of every item
        running = 0;
#pragma unroll
        for (int c = 0; c < kCache + 1; ++c) {
            for (int32_t c0 = c * (int32_t)blockDim.x; c0 < n_seqs; c0 += (c < kCache ? n_seqs : (int32_t)blockDim.x)) {
                const int32_t s = c0 + tid;
                int32_t n = 0, pre = 0, st = 0;
                if (s < n_seqs && chunk > 0) {
                    pre = c < kCache ? ex_c[c] : ws.seq_prefix[s];
                    const int32_t ctx = ctx_of(c, s);
                    st = (ctx < 0 || ctx > max_tokens) ? 0 : (ctx + kStageTokens - 1) / kStageTokens;
                    if (st > 0) n = (pre + st - 1) / chunk - pre / chunk + 1;
                }
                int32_t tot;
                const int32_t ex = running + block_exclusive_scan(n, &tot, scratch);
                if (s < n_seqs) {
                    ws.seg[s] = make_int2(ex, n);
                    // items whose first stage lies in this sequence start with it
                    for (int32_t i = (pre + chunk - 1) / max(chunk, 1); st > 0 && i * chunk < pre + st; ++i)
                        ws.items[i] = make_int2(s, 0);
                }
                running += tot;
            }
        }
    }
    if (tid == 0) {
        if (overflow) report(dev_status, PKV_DEV_WORKSPACE_OVERFLOW);
        ws.header[kHdrTotal] = overflow ? 0u : (uint32_t)n_items;
        ws.header[kHdrOverflow] = overflow ? 1u : 0u;
        ws.header[kHdrChunk] = (uint32_t)chunk;
        ws.header[kHdrStages] = balanced && !overflow ? (uint32_t)total_stages : 0u;
        ws.header[kHdrCounter] = 0u;
    }
    // Sequences no piece will cover (empty or invalid context, or every
    // sequence when the work list overflowed) get o = 0 and lse = -inf here,
    // one thread per such sequence.
#pragma unroll
    for (int c = 0; c < kCache + 1; ++c) {
        for (int32_t c0 = c * (int32_t)blockDim.x; c0 < n_seqs; c0 += (c < kCache ? n_seqs : (int32_t)blockDim.x)) {
            const int32_t s = c0 + tid;
            if (s >= n_seqs) continue;
            const int32_t ctx = ctx_of(c, s);
            if (!overflow && ctx > 0 && ctx <= max_tokens) continue;
            const int64_t row = (int64_t)s * n_q_heads;
            uint4 *o = reinterpret_cast<uint4 *>(out + row * head_dim);
            for (int32_t i = 0; i < n_q_heads * head_dim / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
            if (lse_out)
                for (int32_t i = 0; i < n_q_heads; ++i) lse_out[row + i] = -INFINITY;
        }
    }
}

// ---------------------------------------------------------------------------
// 3. merge of the pieces of a sequence
// ---------------------------------------------------------------------------
// Merge of the pieces of a sequence, per (sequence, query head):
// o = sum_k 2^(m_k - M) acc_k / sum_k 2^(m_k - M) l_k with M = max_k m_k (the
// finalize step of the tiled attention), lse = ln 2 (M + log2 L).  A warp
// merges one (sequence, query head) pair at a time, the pairs of the grid
// taken in a grid-stride loop (the grid is a few CTAs per SM, so no wave of
// short-lived CTAs waits behind another).  Per pair, the pieces go kRound at a
// time: lane i < kRound reads piece k0 + i's (m, l) while every lane reads its
// D / 32 elements of the round's partial rows, all in flight together (a pair
// of up to kRound pieces costs one memory round trip); the round's maximum
// rescales the running sums (an online merge) and each row is weighted by its
// piece's factor broadcast from the lane that read it.  Partials are read with
// ld.global.cg (L2: other SMs wrote them), marked to be evicted first; with
// drop_partials (fixed splits, whose partials grow with the context) a pair's
// rows are then discarded from L2, so the dead lines are never written back.
// Launched after the split kernel as a programmatic dependent: the plan's
// results are complete when it starts (the split kernel releases it only after
// its own wait for the plan); only the partials need the wait for the split
// kernel.
constexpr int kMergeCtasPerSm = 6;

template <int D>
__global__ void __launch_bounds__(128, kMergeCtasPerSm) decode_merge_kernel(DecodeWorkspace ws, int32_t n_seqs,
                                                                           int32_t n_q_heads, __nv_bfloat16 *out,
                                                                           float *lse_out, int32_t drop_partials)
{
    constexpr int EPL = D / 32;                      // output elements per lane
    constexpr int kRound = 8;                        // pieces per round
    grid_dependents_launch();   // the next step's plan may start; it waits for this grid
    const int lane = threadIdx.x & 31;
    const int64_t n_pairs = (int64_t)n_seqs * n_q_heads;
    const int64_t n_warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t idx0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    // the plan's results are read before the wait: the first pair's pieces
    // (with one pair per warp, the only ones) and the overflow flag
    const uint32_t overflow = ws.header[kHdrOverflow];
    const int2 sg0 = idx0 < n_pairs ? ws.seg[idx0 / n_q_heads] : make_int2(0, 0);
    grid_dependency_wait();
    if (overflow != 0) return;
    const uint64_t drop = l2_evict_first_policy();
    for (int64_t idx = idx0; idx < n_pairs; idx += n_warps) {
        const int32_t s = (int32_t)(idx / n_q_heads), h = (int32_t)(idx % n_q_heads);
        const int2 sg = idx == idx0 ? sg0 : ws.seg[s];
        if (sg.y < 2) continue;
        const int32_t n = sg.y;
        const int64_t row0 = (int64_t)sg.x * n_q_heads + h;   // piece k's row: row0 + k * n_q_heads
        const int64_t stride = (int64_t)n_q_heads * D;         // floats from one piece's row to the next
        const float *base = ws.part_acc + row0 * D + lane * EPL;
        float M = -INFINITY, Lsum = 0.f;                       // Lsum: lanes < kRound, scaled to 2^-M
        float o[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[e] = 0.f;
        for (int32_t k0 = 0; k0 < n; k0 += kRound) {
            const int32_t cnt = min(kRound, n - k0);
            const float2 ml = lane < cnt ? ld_last_use(&ws.part_ml[row0 + (int64_t)(k0 + lane) * n_q_heads], drop)
                                         : make_float2(-INFINITY, 0.f);
            float a[kRound][EPL];
#pragma unroll
            for (int i = 0; i < kRound; ++i) {
                if (i < cnt) {
                    const float *src = base + (int64_t)(k0 + i) * stride;
                    if constexpr (EPL == 4) {
                        const float4 x = ld_last_use(reinterpret_cast<const float4 *>(src), drop);
                        a[i][0] = x.x;
                        a[i][1] = x.y;
                        a[i][2] = x.z;
                        a[i][3] = x.w;
                    } else {
                        const float2 x = ld_last_use(reinterpret_cast<const float2 *>(src), drop);
                        a[i][0] = x.x;
                        a[i][1] = x.y;
                    }
                }
            }
            float mr = ml.x;
#pragma unroll
            for (int off = kRound / 2; off > 0; off >>= 1) mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, off));
            mr = __shfl_sync(0xffffffffu, mr, 0);        // lanes >= kRound held -inf
            const float Mn = fmaxf(M, mr);
            if (Mn != -INFINITY && Mn != M) {             // the maximum moved: rescale what was summed
                const float alpha = exp2f(M - Mn);        // M = -inf gives 0 (nothing summed yet)
                Lsum *= alpha;
#pragma unroll
                for (int e = 0; e < EPL; ++e) o[e] *= alpha;
                M = Mn;
            }
            const float wk = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
            Lsum += wk * ml.y;
#pragma unroll
            for (int i = 0; i < kRound; ++i) {
                const float w = __shfl_sync(0xffffffffu, wk, i);
                if (i < cnt) {
#pragma unroll
                    for (int e = 0; e < EPL; ++e) o[e] = fmaf(w, a[i][e], o[e]);
                }
            }
        }
#pragma unroll
        for (int off = kRound / 2; off > 0; off >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, off);
        Lsum = __shfl_sync(0xffffffffu, Lsum, 0);
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
        __nv_bfloat16 *dst = out + ((int64_t)s * n_q_heads + h) * D + lane * EPL;
        if constexpr (EPL == 4)
            *reinterpret_cast<uint2 *>(dst) =
                make_uint2(pack_bf16x2(o[0] * inv, o[1] * inv), pack_bf16x2(o[2] * inv, o[3] * inv));
        else
            *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(o[0] * inv, o[1] * inv);
        if (lse_out && lane == 0)
            lse_out[(int64_t)s * n_q_heads + h] =
                Lsum > 0.f ? (M + __log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
        // the pair's partial rows are dead (every lane has used its values):
        // their L2 lines are dropped without a write-back, lane l taking lines
        // l, l + 32, ... (row i / LINES, line i % LINES)
        if (drop_partials) {
            __syncwarp();
            constexpr int LINES = D / 32;   // 128-byte lines per row of D floats
            for (int i = lane; i < n * LINES; i += 32)
                l2_discard_line(ws.part_acc + (row0 + (int64_t)(i / LINES) * n_q_heads) * D + (i % LINES) * 32);
        }
    }
}

// TMA copies of one 16-token stage (K and V tiles of hpc kv heads, int8 scales)
template <int D, bool INT8>
__device__ __forceinline__ void issue_stage_loads(uint8_t *stg, const DecodeParams &p, const CUtensorMap &k_map,
                                                  const CUtensorMap &v_map, const CUtensorMap &ks_map,
                                                  const CUtensorMap &vs_map, int32_t row0, int32_t head0,
                                                  uint64_t *bar)
{
    constexpr int HALVES = D / 64;
    if (!INT8) {
        const uint32_t half_bytes = (uint32_t)p.hpc * kStageTokens * 128u;
        for (int h = 0; h < HALVES; ++h) {
            for (int b = 0; b < p.boxes_per_half; ++b) {
                const uint32_t off = h * half_bytes + b * (kStageTokens * 128u);
                if (p.boxes_per_half == 1) {
                    tma_load_3d(stg + off, &k_map, h * 64, row0, head0, bar);
                    tma_load_3d(stg + p.kv_tile_bytes + off, &v_map, h * 64, row0, head0, bar);
                } else {
                    tma_load_3d(stg + off, &k_map, h * 64, head0 + b, row0, bar);
                    tma_load_3d(stg + p.kv_tile_bytes + off, &v_map, h * 64, head0 + b, row0, bar);
                }
            }
        }
    } else {
        for (int b = 0; b < p.boxes_per_half; ++b) {
            const uint32_t off = b * (kStageTokens * (uint32_t)D);
            if (p.boxes_per_half == 1) {
                tma_load_3d(stg + off, &k_map, 0, row0, head0, bar);
                tma_load_3d(stg + p.kv_tile_bytes + off, &v_map, 0, row0, head0, bar);
            } else {
                tma_load_3d(stg + off, &k_map, 0, head0 + b, row0, bar);
                tma_load_3d(stg + p.kv_tile_bytes + off, &v_map, 0, head0 + b, row0, bar);
            }
        }
        // the scale box starts at a multiple of scale_heads heads (its first
        // coordinate times 4 bytes must be a multiple of 16)
        if (p.scales_in_stage) {
            uint8_t *sc = stg + 2 * p.kv_tile_bytes;
            const int32_t sh0 = head0 / p.scale_heads * p.scale_heads;
            tma_load_2d(sc, &ks_map, sh0, row0, bar);
            tma_load_2d(sc + p.scale_tile_bytes, &vs_map, sh0, row0, bar);
        }
    }
}

// The producer of the split kernels (one thread): walks this CTA's units of
// the work list, streams their pages stage by stage into the ring and ends it
// with a stop marker.
template <int D, bool INT8>
__device__ __forceinline__ void run_producer(const SmemLayout &L, const DecodeParams &p, const CUtensorMap &k_map,
                                             const CUtensorMap &v_map, const CUtensorMap &ks_map,
                                             const CUtensorMap &vs_map, volatile int32_t *abort_flag,
                                             uint32_t total_items)
{
    const int hpc = p.hpc;
    // ===================== producer (one thread) =====================
    // Lane 0 alone walks the work list and issues the copies: no per-stage
    // warp shuffles or divergent branches, ring position and block
    // position advanced by counters, the next table entry loaded one stage
    // ahead of its use.
    prefetch_tensormap(&k_map);
    prefetch_tensormap(&v_map);
    if (INT8) {
        prefetch_tensormap(&ks_map);
        prefetch_tensormap(&vs_map);
    }
    uint32_t st = 0, phase = 0;          // ring slot and its parity
    uint32_t item_it = 0;
    bool ok = true;
    const bool balanced = p.split_tokens == 0;
    const int32_t chunk = (int32_t)p.ws.header[kHdrChunk];
    const int32_t total_stages = (int32_t)p.ws.header[kHdrStages];
    // Balanced items are all the same size and number at most the grid:
    // CTA b takes units b, b + grid, ...  Fixed splits differ in size: a
    // CTA takes the next unit from the counter when it starts one (no id
    // is taken ahead, which would let early CTAs hold two units while late
    // ones get none).
    uint32_t it = balanced ? blockIdx.x : atomicAdd(&p.ws.header[kHdrCounter], 1u);
    for (; ok && it < total_items;
         it = balanced ? it + gridDim.x : atomicAdd(&p.ws.header[kHdrCounter], 1u)) {
        const int32_t item = (int32_t)(it / p.n_hg), hg = (int32_t)(it % p.n_hg);
        // balanced: the item is the stage range [g0, g1) of the concatenated sequences
        int32_t g0 = 0, g1 = 0, sq = 0;
        int2 fixed_sk = make_int2(0, 0);
        if (balanced) {
            g0 = item * chunk;
            g1 = min(g0 + chunk, total_stages);
            sq = __ldg(&p.ws.items[item].x);
        } else {
            fixed_sk = __ldg(&p.ws.items[item]);
        }
        bool more = true;
        while (ok && more) {
            // the next piece: sequence, token range, partial slot, pieces of that sequence
            int32_t seq, t0, t1, slot, n_pieces;
            if (balanced) {
                int32_t pre = __ldg(p.ws.seq_prefix + sq), pre1 = __ldg(p.ws.seq_prefix + sq + 1);
                while (pre1 == pre) {  // sequences without tokens
                    ++sq;
                    pre = pre1;
                    pre1 = __ldg(p.ws.seq_prefix + sq + 1);
                }
                const int32_t e = min(g1, pre1);
                seq = sq;
                t0 = (g0 - pre) * kStageTokens;
                t1 = min((e - pre) * kStageTokens, __ldg(p.ctx_lens + sq));
                const int2 sg = __ldg(p.ws.seg + sq);
                slot = sg.x + (item - pre / chunk);
                n_pieces = sg.y;
                g0 = e;
                ++sq;
                more = g0 < g1;
            } else {
                seq = fixed_sk.x;
                t0 = fixed_sk.y * p.split_tokens;
                t1 = min(t0 + p.split_tokens, __ldg(p.ctx_lens + seq));
                slot = item;
                n_pieces = __ldg(&p.ws.seg[seq].y);
                more = false;
            }
            const bool final_out = n_pieces == 1;
            const int32_t *trow = p.tables + (int64_t)seq * p.max_blocks;
            // this piece's queries: heads [hg*hpc*G, (hg+1)*hpc*G) of sequence seq
            const uint32_t qs = item_it & 1u;
            if (!mbar_wait(&L.qempty_bar[qs], ((item_it >> 1) & 1u) ^ 1u, abort_flag, p.wait_ns)) {
                report(p.dev_status, PKV_DEV_TIMEOUT);
                *abort_flag = 1;
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(&L.qfull_bar[qs], p.q_slot_bytes);
            bulk_g2s(L.q_slots + qs * p.q_slot_bytes,
                     p.q + ((int64_t)seq * p.n_q_heads + (int64_t)hg * hpc * p.group) * D, p.q_slot_bytes,
                     &L.qfull_bar[qs]);
            // block position of t0, and its table entry; later entries are
            // loaded one stage ahead
            int32_t lb = t0 / p.block_size, off = t0 - lb * p.block_size;
            int32_t blk = lb < p.max_blocks ? __ldg(trow + lb) : -1;
            for (int32_t t = t0; t < t1; t += kStageTokens) {
                const bool last_of_block = off + kStageTokens >= p.block_size;
                const bool more_stages = t + kStageTokens < t1;
                int32_t blk_next = blk;
                if (last_of_block && more_stages) blk_next = lb + 1 < p.max_blocks ? __ldg(trow + lb + 1) : -1;
                if (!mbar_wait(&L.empty_bar[st], phase ^ 1u, abort_flag, p.wait_ns)) {
                    report(p.dev_status, PKV_DEV_TIMEOUT);
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
                StageMeta m;
                m.seq = seq;
                m.split_index = slot;
                m.n_valid = min(kStageTokens, t1 - t);
                m.flags = (t == t0 ? kMetaFirst : 0) | (more_stages ? 0 : kMetaLast) | (final_out ? kMetaFinal : 0);
                m.head_group = hg;
                m.n_splits = n_pieces;
                const bool bad = blk < 0 || blk > p.n_blocks;
                if (bad) {
                    m.flags |= kMetaBad;
                    report(p.dev_status, PKV_DEV_BAD_BLOCK_ID);
                }
                const int32_t row0 = bad ? 0 : blk * p.block_size + off;
                m.row0 = row0;
                m.pad = 0;
                L.meta[st] = m;
                if (bad) {
                    mbar_arrive(&L.full_bar[st]);
                } else {
                    uint8_t *stg = L.stages + (size_t)st * p.stage_bytes;
                    mbar_arrive_expect_tx(&L.full_bar[st], p.tx_bytes);
                    issue_stage_loads<D, INT8>(stg, p, k_map, v_map, ks_map, vs_map, row0, hg * hpc,
                                               &L.full_bar[st]);
                }
                if (++st == (uint32_t)p.n_stages) {
                    st = 0;
                    phase ^= 1u;
                }
                if (last_of_block) {
                    ++lb;
                    off = 0;
                    blk = blk_next;
                } else {
                    off += kStageTokens;
                }
            }
            if (ok && p.tile_stages > 1) {
                // the tensor-core kernel takes whole tiles of tile_stages stages:
                // the piece is padded with empty stages up to the next tile
                const int32_t used = (t1 - t0 + kStageTokens - 1) / kStageTokens;
                for (int32_t k = (p.tile_stages - used % p.tile_stages) % p.tile_stages; k > 0; --k) {
                    if (!mbar_wait(&L.empty_bar[st], phase ^ 1u, abort_flag, p.wait_ns)) {
                        report(p.dev_status, PKV_DEV_TIMEOUT);
                        *abort_flag = 1;
                        ok = false;
                        break;
                    }
                    L.meta[st].flags = kMetaPad;
                    mbar_arrive(&L.full_bar[st]);
                    if (++st == (uint32_t)p.n_stages) {
                        st = 0;
                        phase ^= 1u;
                    }
                }
            }
            ++item_it;
        }
    }
    // stop marker
    if (ok && !*abort_flag) {
        if (mbar_wait(&L.empty_bar[st], phase ^ 1u, abort_flag, p.wait_ns)) {
            L.meta[st].flags = kMetaStop;
            mbar_arrive(&L.full_bar[st]);
        } else {
            report(p.dev_status, PKV_DEV_TIMEOUT);
            *abort_flag = 1;
        }
    }
    if (*abort_flag) {
        // wind down: let every copy already issued land before the CTA exits
        // (the last n_stages slots and the last two query copies; a phase
        // never issued counts as complete), with the default limit
        uint32_t ws_ = st, wp = phase;
        for (int i = 0; i < p.n_stages; ++i) {
            if (ws_ == 0) {
                ws_ = (uint32_t)p.n_stages;
                wp ^= 1u;
            }
            --ws_;
            (void)mbar_wait(&L.full_bar[ws_], wp);
        }
        for (uint32_t i = item_it > 2u ? item_it - 2u : 0u; i < item_it; ++i)
            (void)mbar_wait(&L.qfull_bar[i & 1u], (i >> 1) & 1u);
    }
}

// ---------------------------------------------------------------------------
// 2. split kernel
// ---------------------------------------------------------------------------
// Register budget (measured on GB300): bf16 pages compile for two resident
// 288-thread CTAs per SM (at most ~112 registers; fewer registers measured
// faster even at one CTA per SM), int8 pages for one (the fp16 fragments of the
// in-register code conversion need ~168 registers; the two-CTA budget spills).
// int8 pages launch 160-thread CTAs (four kv heads), two of which fit an SM at
// that register count.
template <int D, bool INT8>
__global__ void __launch_bounds__(288, INT8 ? 1 : 2) decode_split_kernel(const __grid_constant__ CUtensorMap k_map,
                                                              const __grid_constant__ CUtensorMap v_map,
                                                              const __grid_constant__ CUtensorMap ks_map,
                                                              const __grid_constant__ CUtensorMap vs_map,
                                                              const DecodeParams p)
{
    constexpr int KSTEPS = D / 16;      // mma k-steps over head_dim (QK) = m-tiles (PV)
    extern __shared__ uint8_t smem_raw[];
    SmemLayout L = carve(smem_raw, p);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hpc = p.hpc;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.n_stages; ++i) {
            mbar_init(&L.full_bar[i], 1);
            mbar_init(&L.empty_bar[i], hpc);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&L.qfull_bar[i], 1);
            mbar_init(&L.qempty_bar[i], hpc);
        }
        *L.abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    grid_dependency_wait();     // the plan kernel's work list is complete and visible
    // the merge may start now: the plan it reads first is complete
    grid_dependents_launch();

    const uint32_t total_items = p.ws.header[kHdrTotal] * (uint32_t)p.n_hg;
    volatile int32_t *abort_flag = L.abort_flag;

    if (warp == hpc) {
        if (lane == 0) run_producer<D, INT8>(L, p, k_map, v_map, ks_map, vs_map, abort_flag, total_items);
        return;
    }
    if (warp > hpc) return;

    // ===================== consumer warps (one kv head each) =====================
    const int g = lane >> 2, qd = lane & 3;   // mma fragment row group / column pair
    const int G = p.group;
    const int mi = lane >> 3, ri = lane & 7;  // ldmatrix matrix index / row within it
    float acc[KSTEPS][4];                     // O^T accumulators: rows d, columns query heads
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    // int8 pages: bias corrections of this lane's columns n0 = 2qd, n1 = 2qd + 1
    // (qb: 1152 * sum_d q_d of the piece's query heads; ps: running sum of
    // the fp16 P' fed to the P V product, rescaled with acc)
    float qb0 = 0.f, qb1 = 0.f, ps0 = 0.f, ps1 = 0.f;
    uint32_t st = 0, phase = 0, item_it = 0;   // ring slot and its parity
    const uint32_t half_bytes = (uint32_t)hpc * kStageTokens * 128u;

    while (true) {
        if (!__all_sync(0xffffffffu, mbar_wait(&L.full_bar[st], phase, abort_flag, p.wait_ns))) {
            if (lane == 0) report(p.dev_status, PKV_DEV_TIMEOUT);
            *abort_flag = 1;
            break;
        }
        const StageMeta meta = L.meta[st];
        if (meta.flags & kMetaStop) break;
        uint8_t *stg = L.stages + (size_t)st * p.stage_bytes;

        if (meta.flags & kMetaFirst) {
            const uint32_t qs = item_it & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait(&L.qfull_bar[qs], (item_it >> 1) & 1u, abort_flag, p.wait_ns))) {
                if (lane == 0) report(p.dev_status, PKV_DEV_TIMEOUT);
                *abort_flag = 1;
                break;
            }
            // Rewrite this warp's G query rows in place: 16-byte chunk c of head row
            // r moves to chunk c ^ r (so ldmatrix of 8 head rows is conflict-free).
            // For int8 pages the row is also converted to fp16 and its elements
            // permuted so that k-step kk, lane q of the K^T Q contraction sees
            // d = q * D/4 + 4 kk + {0, 1} (b0) and + {2, 3} (b1): the order in
            // which each lane holds its K codes (a dot product does not depend
            // on the order of its terms).  The rows stay in the slot until the
            // piece's last stage.
            uint8_t *qrows = L.q_slots + qs * p.q_slot_bytes + (size_t)warp * G * D * 2;
            {
                constexpr int CPR = D / 8;            // 16-byte chunks per head row
                uint4 tmp[(8 * CPR + 31) / 32];
#pragma unroll
                for (int i = 0; i < (8 * CPR + 31) / 32; ++i) {
                    const int idx = i * 32 + lane;
                    if (idx < G * CPR) {
                        if (!INT8) {
                            tmp[i] = *reinterpret_cast<const uint4 *>(qrows + idx * 16);
                        } else {
                            const int r = idx / CPR, c = idx % CPR, kk = c / 2, h = c % 2;
                            uint32_t *w = reinterpret_cast<uint32_t *>(&tmp[i]);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const int d0 = q * (D / 4) + 4 * kk + 2 * h;
                                const uint32_t bits = *reinterpret_cast<const uint32_t *>(qrows + (r * D + d0) * 2);
                                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&bits));
                                w[q] = pack_f16x2(f.x, f.y);
                            }
                        }
                    }
                }
                __syncwarp();
#pragma unroll
                for (int i = 0; i < (8 * CPR + 31) / 32; ++i) {
                    const int idx = i * 32 + lane;
                    if (idx < G * CPR) {
                        const int r = idx / CPR, c = idx % CPR;
                        *reinterpret_cast<uint4 *>(qrows + (r * CPR + (c ^ (r & 7))) * 16) = tmp[i];
                    }
                }
                __syncwarp();
            }
            if (INT8) {
                // sum_d q_d of the fp16 query rows of columns n0, n1 (padding
                // columns read row 0): lane (g, qd) adds its share of the
                // chunks (the swizzle only permutes chunks within a row)
                constexpr int CPR = D / 8;
                const int r0 = 2 * qd < G ? 2 * qd : 0, r1 = 2 * qd + 1 < G ? 2 * qd + 1 : 0;
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int c = g; c < CPR; c += 8) {
                    const uint4 x0 = *reinterpret_cast<const uint4 *>(qrows + (r0 * CPR + c) * 16);
                    const uint4 x1 = *reinterpret_cast<const uint4 *>(qrows + (r1 * CPR + c) * 16);
                    const uint32_t w0[4] = {x0.x, x0.y, x0.z, x0.w}, w1[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&w0[k]));
                        const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&w1[k]));
                        a0 += f0.x + f0.y;
                        a1 += f1.x + f1.y;
                    }
                }
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    a0 += __shfl_xor_sync(0xffffffffu, a0, off);
                    a1 += __shfl_xor_sync(0xffffffffu, a1, off);
                }
                qb0 = kCodeBias * a0;
                qb1 = kCodeBias * a1;
                ps0 = ps1 = 0.f;
            }
#pragma unroll
            for (int mt = 0; mt < KSTEPS; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
        }

        if (!(meta.flags & kMetaBad)) {
            const int nv = meta.n_valid;
            // --- tiles for this head: bf16 through ldmatrix; int8 codes are read
            // straight into mma fragments
            uint32_t k_base, v_base;     // smem address of half 0 of this head's K / V tile
            uint32_t half_stride;        // bytes between the two 64-column halves
            float sk0 = 1.f, sk1 = 1.f, sv0 = 1.f, sv1 = 1.f;
            const uint8_t *kcodes = stg + (size_t)warp * kStageTokens * D;   // int8: this head's codes
            if (!INT8) {
                k_base = smem_u32(stg) + warp * (kStageTokens * 128u);
                v_base = k_base + p.kv_tile_bytes;
                half_stride = half_bytes;
            } else {
                k_base = v_base = half_stride = 0;
                const float *sc = reinterpret_cast<const float *>(stg + 2 * p.kv_tile_bytes);
                sk0 = sc[g * hpc + warp];
                sk1 = sc[(g + 8) * hpc + warp];
                const float *scv = sc + p.scale_tile_bytes / 4;
                sv0 = scv[g * hpc + warp];
                sv1 = scv[(g + 8) * hpc + warp];
            }

            // --- S^T[16 tokens x 8 heads] = K Q^T; Q^T B-fragments by ldmatrix from the
            // swizzled query rows.  Padding columns (heads G..7) re-read row 0 of
            // this warp: their results are never used, and every address stays
            // inside this warp's G rows of the slot.
            const uint32_t q_base = smem_u32(L.q_slots + (item_it & 1u) * p.q_slot_bytes) + warp * G * D * 2;
            const uint32_t qrow = ri < G ? (uint32_t)ri : 0u;
            float s4[4] = {0.f, 0.f, 0.f, 0.f};
            // int8: lane (g, qd) holds the D/4 codes d = qd * D/4 .. of token rows g and
            // g + 8 (one or two conflict-free 16-byte loads per row); word kk of
            // that run is k-step kk's A fragment (a0a1 | a4a5 from row g, a2a3 |
            // a6a7 from row g + 8), converted exactly to fp16.
            uint32_t kw[2][D / 16];
            if (INT8) {
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const int tok = g + 8 * rr;
#pragma unroll
                    for (int c = 0; c < D / 64; ++c) {
                        const uint32_t off = D == 128 ? swz(tok, 2 * qd + c) : (uint32_t)(tok * D + qd * 16);
                        const uint4 x = *reinterpret_cast<const uint4 *>(kcodes + off);
                        kw[rr][4 * c] = x.x;
                        kw[rr][4 * c + 1] = x.y;
                        kw[rr][4 * c + 2] = x.z;
                        kw[rr][4 * c + 3] = x.w;
                    }
                }
            }
            // int8: V codes for O^T += V^T P^T, loaded and converted (biased) up
            // front so the conversion overlaps the K Q^T chain.  Lane (g, qd) holds
            // the D/8 codes d = g * D/8 .. of tokens 2qd, 2qd+1, 2qd+8, 2qd+9;
            // O^T rows are relabelled: m-tile mt row g is d = g * D/8 + 2 mt and
            // row g + 8 is the next d, so byte pairs of two token rows interleave
            // (prmt) into the A fragments.
            uint32_t va[INT8 ? KSTEPS : 1][4];
            if constexpr (INT8) {
                uint32_t vw[4][D / 32];
#pragma unroll
                for (int t4 = 0; t4 < 4; ++t4) {
                    const int tok = 2 * qd + (t4 & 1) + 8 * (t4 >> 1);
                    if (D == 128) {
                        const uint4 x = *reinterpret_cast<const uint4 *>(kcodes + p.kv_tile_bytes + swz(tok, g));
                        vw[t4][0] = x.x;
                        vw[t4][1] = x.y;
                        vw[t4][2] = x.z;
                        vw[t4][3] = x.w;
                    } else {
                        const uint2 x = *reinterpret_cast<const uint2 *>(kcodes + p.kv_tile_bytes + tok * D + g * 8);
                        vw[t4][0] = x.x;
                        vw[t4][1] = x.y;
                    }
                }
#pragma unroll
                for (int mt = 0; mt < KSTEPS; ++mt) {
                    const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
                    int8x4_to_biased_half2x2(__byte_perm(vw[0][mt / 2], vw[1][mt / 2], sel), va[mt][0], va[mt][1]);
                    int8x4_to_biased_half2x2(__byte_perm(vw[2][mt / 2], vw[3][mt / 2], sel), va[mt][2], va[mt][3]);
                }
            }
            // K Q^T; int8 pages in two accumulator chains (even and odd k-steps)
            float s4b[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < KSTEPS; kk += 2) {
                uint32_t qb[4];  // b0, b1 of k-step kk, then of kk + 1
                ldmatrix_x4(qb, q_base + qrow * (D * 2) + (((uint32_t)(2 * kk + mi) ^ (qrow & 7u)) << 4));
#pragma unroll
                for (int k2 = 0; k2 < 2; ++k2) {
                    const int k = kk + k2;
                    uint32_t a[4];
                    if constexpr (INT8) {
                        int8x4_to_biased_half2x2(kw[0][k], a[0], a[2]);
                        int8x4_to_biased_half2x2(kw[1][k], a[1], a[3]);
                        mma_f16_16816(k2 ? s4b : s4, a, qb[2 * k2], qb[2 * k2 + 1]);
                    } else {
                        const int tok = ri + 8 * (mi & 1);
                        const uint32_t chunk = (uint32_t)((k % 4) * 2 + (mi >> 1));
                        ldmatrix_x4(a, k_base + (uint32_t)(k / 4) * half_stride + swz(tok, chunk));
                        mma_bf16_16816(s4, a, qb[2 * k2], qb[2 * k2 + 1]);
                    }
                }
            }
            // scale to log2 units, dequantise K (int8: remove the code bias
            // 1152 sum_d q_d first), mask tokens past the context
            const bool v0 = g < nv, v1 = g + 8 < nv;
            float x0, x1, x2, x3;
            if constexpr (INT8) {
                const float c0 = sk0 * p.scale_log2, c1 = sk1 * p.scale_log2;
                x0 = v0 ? ((s4[0] + s4b[0]) - qb0) * c0 : -INFINITY;
                x1 = v0 ? ((s4[1] + s4b[1]) - qb1) * c0 : -INFINITY;
                x2 = v1 ? ((s4[2] + s4b[2]) - qb0) * c1 : -INFINITY;
                x3 = v1 ? ((s4[3] + s4b[3]) - qb1) * c1 : -INFINITY;
            } else {
                x0 = v0 ? s4[0] * p.scale_log2 : -INFINITY;
                x1 = v0 ? s4[1] * p.scale_log2 : -INFINITY;
                x2 = v1 ? s4[2] * p.scale_log2 : -INFINITY;
                x3 = v1 ? s4[3] * p.scale_log2 : -INFINITY;
            }
            // Lazy running maximum (log2 units): it moves only when a score of
            // the stage passes it by more than kLazyMax, so the probabilities
            // stay at most 2^kLazyMax, and the row reduction and the rescale of
            // the accumulators run only then (o = acc / l and lse = m + log2 l
            // do not depend on which m was used).
            if (__any_sync(0xffffffffu, fmaxf(x0, x2) > m0 + kLazyMax || fmaxf(x1, x3) > m1 + kLazyMax)) {
                float bm0 = fmaxf(x0, x2), bm1 = fmaxf(x1, x3);
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, off));
                    bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, off));
                }
                const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
                const float al0 = fast_exp2(m0 - mn0), al1 = fast_exp2(m1 - mn1);
                m0 = mn0;
                m1 = mn1;
                l0 *= al0;
                l1 *= al1;
#pragma unroll
                for (int mt = 0; mt < KSTEPS; ++mt) {
                    acc[mt][0] *= al0;
                    acc[mt][1] *= al1;
                    acc[mt][2] *= al0;
                    acc[mt][3] *= al1;
                }
                ps0 *= al0;
                ps1 *= al1;
            }
            const float p0 = fast_exp2(x0 - m0), p1 = fast_exp2(x1 - m1);
            const float p2 = fast_exp2(x2 - m0), p3 = fast_exp2(x3 - m1);
            l0 += p0 + p2;
            l1 += p1 + p3;
            // P^T as the B operand of O^T += V^T P^T (int8: fold the V scale into
            // P, and add the fp16 P' actually used to the bias correction's sum)
            uint32_t pb0, pb1;
            if constexpr (INT8) {
                const uint32_t pk0 = pack_f16x2(v0 ? p0 * sv0 : 0.f, v0 ? p1 * sv0 : 0.f);
                const uint32_t pk1 = pack_f16x2(v1 ? p2 * sv1 : 0.f, v1 ? p3 * sv1 : 0.f);
                const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&pk0));
                const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&pk1));
                ps0 += f0.x + f1.x;
                ps1 += f0.y + f1.y;
                pb0 = movmatrix_trans(pk0);
                pb1 = movmatrix_trans(pk1);
#pragma unroll
                for (int mt = 0; mt < KSTEPS; ++mt) mma_f16_16816(acc[mt], va[mt], pb0, pb1);
            } else {
                pb0 = movmatrix_trans(pack_bf16x2(p0, p1));
                pb1 = movmatrix_trans(pack_bf16x2(p2, p3));
                // V rows past the context may hold anything (even NaN): zero them in
                // the A fragments of a partial stage so 0 * NaN never reaches the sum.
                uint32_t vmask0 = 0xffffffffu, vmask1 = 0xffffffffu;
                if (nv < kStageTokens) {
                    const int ta = 2 * qd, tb = 2 * qd + 8;
                    vmask0 = (ta < nv ? 0x0000ffffu : 0u) | (ta + 1 < nv ? 0xffff0000u : 0u);
                    vmask1 = (tb < nv ? 0x0000ffffu : 0u) | (tb + 1 < nv ? 0xffff0000u : 0u);
                }
#pragma unroll
                for (int mt = 0; mt < KSTEPS; ++mt) {
                    const int tok = ri + 8 * (mi >> 1);
                    const uint32_t chunk = (uint32_t)((mt % 4) * 2 + (mi & 1));
                    uint32_t a[4];
                    ldmatrix_x4_trans(a, v_base + (uint32_t)(mt / 4) * half_stride + swz(tok, chunk));
                    a[0] &= vmask0;
                    a[1] &= vmask0;
                    a[2] &= vmask1;
                    a[3] &= vmask1;
                    mma_bf16_16816(acc[mt], a, pb0, pb1);
                }
            }
            (void)va;
        }

        // the stage's tiles (and, at a piece's end, its query rows) are no longer
        // needed: hand them back before finalising
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&L.empty_bar[st]);
            if (meta.flags & kMetaLast) mbar_arrive(&L.qempty_bar[item_it & 1u]);
        }
        if (++st == (uint32_t)p.n_stages) {
            st = 0;
            phase ^= 1u;
        }

        if (meta.flags & kMetaLast) {
            float L0 = l0, L1 = l1;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                L0 += __shfl_xor_sync(0xffffffffu, L0, off);
                L1 += __shfl_xor_sync(0xffffffffu, L1, off);
            }
            if constexpr (INT8) {
                // remove the code bias: O^T = (V + 1152)^T P'^T - 1152 sum_t P'_t
                float P0 = ps0, P1 = ps1;
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    P0 += __shfl_xor_sync(0xffffffffu, P0, off);
                    P1 += __shfl_xor_sync(0xffffffffu, P1, off);
                }
                const float B0 = kCodeBias * P0, B1 = kCodeBias * P1;
#pragma unroll
                for (int mt = 0; mt < KSTEPS; ++mt) {
                    acc[mt][0] -= B0;
                    acc[mt][1] -= B1;
                    acc[mt][2] -= B0;
                    acc[mt][3] -= B1;
                }
            }
            const int32_t s = meta.seq;
            const int32_t kvh = meta.head_group * hpc + warp;
            // first query head of this warp's group: columns 2qd, 2qd+1 are hbase + n0, n1
            const int32_t hbase = kvh * G;
            const int n0 = 2 * qd, n1 = 2 * qd + 1;
            if (meta.flags & kMetaFinal) {
                const float inv0 = 1.f / L0, inv1 = 1.f / L1;
                __nv_bfloat16 *o = p.out + ((int64_t)s * p.n_q_heads + hbase) * D;
#pragma unroll
                for (int mt = 0; mt < KSTEPS; ++mt) {
                    if (INT8) {  // rows g, g + 8 of m-tile mt are d, d + 1
                        const int d = g * (D / 8) + 2 * mt;
                        if (n0 < G)
                            *reinterpret_cast<uint32_t *>(o + (size_t)n0 * D + d) =
                                pack_bf16x2(acc[mt][0] * inv0, acc[mt][2] * inv0);
                        if (n1 < G)
                            *reinterpret_cast<uint32_t *>(o + (size_t)n1 * D + d) =
                                pack_bf16x2(acc[mt][1] * inv1, acc[mt][3] * inv1);
                    } else {     // rows g, g + 8 of m-tile mt are d, d + 8
                        const int d = mt * 16 + g;
                        if (n0 < G) {
                            o[(size_t)n0 * D + d] = __float2bfloat16_rn(acc[mt][0] * inv0);
                            o[(size_t)n0 * D + d + 8] = __float2bfloat16_rn(acc[mt][2] * inv0);
                        }
                        if (n1 < G) {
                            o[(size_t)n1 * D + d] = __float2bfloat16_rn(acc[mt][1] * inv1);
                            o[(size_t)n1 * D + d + 8] = __float2bfloat16_rn(acc[mt][3] * inv1);
                        }
                    }
                }
                if (p.lse_out && g == 0) {
                    float *lo = p.lse_out + (int64_t)s * p.n_q_heads + hbase;
                    if (n0 < G) lo[n0] = (m0 + __log2f(L0)) * 0.69314718055994531f;
                    if (n1 < G) lo[n1] = (m1 + __log2f(L1)) * 0.69314718055994531f;
                }
            } else {
                const int64_t prow = (int64_t)meta.split_index * p.n_q_heads + hbase;
                float *pa = p.ws.part_acc + prow * D;
                const uint64_t keep = l2_evict_last_policy();
#pragma unroll
                for (int mt = 0; mt < KSTEPS; ++mt) {
                    if (INT8) {
                        const int d = g * (D / 8) + 2 * mt;
                        if (n0 < G)
                            st_kept(reinterpret_cast<float2 *>(pa + (size_t)n0 * D + d), make_float2(acc[mt][0], acc[mt][2]),
                                    keep);
                        if (n1 < G)
                            st_kept(reinterpret_cast<float2 *>(pa + (size_t)n1 * D + d), make_float2(acc[mt][1], acc[mt][3]),
                                    keep);
                    } else {
                        const int d = mt * 16 + g;
                        if (n0 < G) {
                            st_kept(pa + (size_t)n0 * D + d, acc[mt][0], keep);
                            st_kept(pa + (size_t)n0 * D + d + 8, acc[mt][2], keep);
                        }
                        if (n1 < G) {
                            st_kept(pa + (size_t)n1 * D + d, acc[mt][1], keep);
                            st_kept(pa + (size_t)n1 * D + d + 8, acc[mt][3], keep);
                        }
                    }
                }
                if (g == 0) {
                    if (n0 < G) st_kept(p.ws.part_ml + prow + n0, make_float2(m0, L0), keep);
                    if (n1 < G) st_kept(p.ws.part_ml + prow + n1, make_float2(m1, L1), keep);
                }
            }
            ++item_it;
        }
    }
}

// ---------------------------------------------------------------------------
// 2b. tensor-core split kernel: int8 pages, head_dim 128, up to 8 query heads
//     per kv head (tcgen05 with TMEM accumulators)
// ---------------------------------------------------------------------------
// The same work list, producer and partial slots as decode_split_kernel, two
// kv heads per CTA, and tiles of 128 tokens (eight stages; each piece is
// padded to whole tiles).  Per kv head one warpgroup converts the tile's codes
// to fp16 in shared memory (the exact biased form 1152 + b, corrected once
// per score and once per output as in the mma.sync kernel), and one thread of
// the issuing warp runs the contractions on the 5th-generation tensor cores:
//   S^T = K Q^T    tcgen05.mma M 128 (tokens), N 16 (query heads, padded),
//                  K-major A (the converted K tile) and B (the query rows);
//   O^T += V^T P'  M 128 (head_dim), N 16, A = the converted V tile read
//                  MN-major, B = P' (fp16, written by the softmax threads).
// S^T and O^T live in TMEM (16 columns each per kv head).  Thread t of the
// warpgroup owns token t of S^T (the online softmax over tokens: running
// maximum per query head, shared by the warpgroup's threads, with the lazy
// rule of the mma.sync kernel) and row d = t of O^T at the end of a piece.
constexpr int kTcHeads = 2;                                 // kv heads per CTA
constexpr int kTcTokens = 128;                              // tokens per tile (M of S^T)
constexpr int kTcStages = kTcTokens / kStageTokens;         // stages per tile
constexpr int kTcN = 16;                                    // padded query heads (N: 16 at M 128)
constexpr int kTcMaxGroup = 8;                              // query slots of 8 heads fit beside the tiles
constexpr int kTcThreads = 32 * (4 * kTcHeads + 2);         // warpgroups, producer, issuer
constexpr int kTcProducerWarp = 4 * kTcHeads, kTcIssuerWarp = 4 * kTcHeads + 1;
constexpr uint32_t kTcTmemCols = 64;                        // per head: S^T 16 + O^T 16 columns (32)
constexpr uint32_t kTcKTile = kTcTokens * 128u * 2u;        // fp16 K tile: 2 panels x 128 rows x 128 B
constexpr uint32_t kTcVTile = kTcTokens * 128u * 2u;        // fp16 V tile (MN-major for the product)
constexpr uint32_t kTcQTile = kTcN * 128u * 2u;             // fp16 query rows: 2 panels x 16 rows x 128 B
constexpr uint32_t kTcPTile = kTcN * 128u * 2u;             // P': 2 panels (64 tokens each) x 16 rows x 128 B
constexpr uint32_t kTcRegion = kTcHeads * (kTcKTile + kTcVTile + kTcQTile + kTcPTile);
constexpr uint32_t kTcRedBytes = kTcHeads * 4 * kTcN * 4;   // cross-warp reductions
enum : uint32_t { kTcInfoFirst = 1, kTcInfoStop = 2 };

struct TcSmem {
    uint8_t *kt, *vt, *qt, *pt;   // head 0; head h at + h * size
    float *red;                   // [kTcHeads][4][kTcN]
    uint64_t *conv_full, *s_full, *p_full, *pv_done, *o_free, *fin;
    uint32_t *info;               // [kTcHeads]: the tile's flags, for the issuer
    uint32_t *tmem_base;
};

__device__ __forceinline__ TcSmem tc_carve(const SmemLayout &L)
{
    TcSmem T;
    uint8_t *b = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(L.full_bar) + smem_tail_bytes() + 1023) & ~uintptr_t(1023));
    T.kt = b;
    T.vt = T.kt + kTcHeads * kTcKTile;
    T.qt = T.vt + kTcHeads * kTcVTile;
    T.pt = T.qt + kTcHeads * kTcQTile;
    T.red = reinterpret_cast<float *>(T.pt + kTcHeads * kTcPTile);
    T.conv_full = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(T.red) + kTcRedBytes);
    T.s_full = T.conv_full + kTcHeads;
    T.p_full = T.s_full + kTcHeads;
    T.pv_done = T.p_full + kTcHeads;
    T.o_free = T.pv_done + kTcHeads;
    T.fin = T.o_free + kTcHeads;
    T.info = reinterpret_cast<uint32_t *>(T.fin + 1);
    T.tmem_base = T.info + kTcHeads;
    return T;
}

// Bytes after the (1024-aligned) end of the split kernel's layout.
__host__ __device__ constexpr size_t tc_smem_extra()
{
    return kTcRegion + kTcRedBytes + (5 * kTcHeads + 1) * sizeof(uint64_t) + (kTcHeads + 1) * 4 + 16;
}

// Named barrier of one warpgroup (ids 1 + h) that also returns the OR of a
// predicate over its threads.
__device__ __forceinline__ bool wg_bar_or(uint32_t id, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, 128, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void wg_bar(uint32_t id) { asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory"); }

// Named barrier of one warpgroup returning the AND of a predicate: a wait that
// ran out for some warp ends the loop for the whole warpgroup at the same
// point, so no warp is left at a barrier the others never reach.
__device__ __forceinline__ bool wg_all(uint32_t id, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, 128, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id)
        : "memory");
    return r != 0;
}

__global__ void __launch_bounds__(kTcThreads, 1) decode_tc_kernel(const __grid_constant__ CUtensorMap k_map,
                                                                 const __grid_constant__ CUtensorMap v_map,
                                                                 const __grid_constant__ CUtensorMap ks_map,
                                                                 const __grid_constant__ CUtensorMap vs_map,
                                                                 const DecodeParams p)
{
    constexpr int D = 128;
    extern __shared__ uint8_t smem_raw[];
    SmemLayout L = carve(smem_raw, p);
    TcSmem T = tc_carve(L);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.n_stages; ++i) {
            mbar_init(&L.full_bar[i], 1);
            mbar_init(&L.empty_bar[i], kTcHeads);   // one warp of each warpgroup converts a stage
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&L.qfull_bar[i], 1);
            mbar_init(&L.qempty_bar[i], kTcHeads);
        }
        for (int h = 0; h < kTcHeads; ++h) {
            mbar_init(&T.conv_full[h], 1);
            mbar_init(&T.s_full[h], 1);
            mbar_init(&T.p_full[h], 1);
            mbar_init(&T.pv_done[h], 1);
            mbar_init(&T.o_free[h], 1);
        }
        mbar_init(T.fin, 1);
        *L.abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kTcIssuerWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(T.tmem_base)),
                     "r"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *T.tmem_base;
    grid_dependency_wait();     // the plan kernel's work list is complete and visible
    grid_dependents_launch();   // the merge may start: the plan it reads first is complete

    const uint32_t total_items = p.ws.header[kHdrTotal] * (uint32_t)p.n_hg;
    volatile int32_t *abort_flag = L.abort_flag;
    const int G = p.group;

    if (warp == kTcProducerWarp) {
        if (lane == 0) run_producer<D, true>(L, p, k_map, v_map, ks_map, vs_map, abort_flag, total_items);
    } else if (warp == kTcIssuerWarp) {
        // ===================== MMA issuer (one thread) =====================
        if (lane == 0) {
            const uint32_t idesc_s = umma_idesc_f16(kTcTokens, kTcN, false, false);
            const uint32_t idesc_o = umma_idesc_f16(D, kTcN, true, false);
            bool ok = true;
            uint32_t tile = 0, pieces[kTcHeads] = {};
            while (ok) {
                uint32_t info[kTcHeads];
                for (int h = 0; h < kTcHeads && ok; ++h) {
                    ok = mbar_wait(&T.conv_full[h], tile & 1, abort_flag);
                    info[h] = ok ? T.info[h] : 0u;
                }
                if (!ok || (info[0] & kTcInfoStop)) break;
                tc_fence_after();
                // S^T = K Q^T: k-step kk covers head_dim 16 kk .. 16 kk + 15 (32 bytes of
                // a 128-byte panel row; panels of 64 columns)
                for (int h = 0; h < kTcHeads; ++h) {
                    const uint64_t a0 = umma_desc_sw128(smem_u32(T.kt + h * kTcKTile), 16, 1024);
                    const uint64_t b0 = umma_desc_sw128(smem_u32(T.qt + h * kTcQTile), 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)
                        umma_bf16(tmem + h * 32u, desc_step(a0, (kk / 4) * (kTcTokens * 128u) + (kk % 4) * 32),
                                  desc_step(b0, (kk / 4) * (kTcN * 128u) + (kk % 4) * 32), idesc_s, kk > 0);
                    umma_commit(&T.s_full[h]);
                }
                // O^T += V^T P': k-step kk covers tokens 16 kk .. 16 kk + 15 (V: group kk of
                // 4 KiB, 64-column panels 2 KiB apart, 8-token halves 1 KiB apart; P': 32
                // bytes of a row, panels of 64 tokens)
                for (int h = 0; h < kTcHeads && ok; ++h) {
                    ok = mbar_wait(&T.p_full[h], tile & 1, abort_flag);
                    const bool first = (info[h] & kTcInfoFirst) != 0;
                    // the first product of a piece overwrites O^T: the warpgroup has read
                    // out the previous piece's
                    if (ok && first && pieces[h] > 0) ok = mbar_wait(&T.o_free[h], (pieces[h] - 1) & 1, abort_flag);
                    if (!ok) break;
                    if (first) ++pieces[h];
                    tc_fence_after();
                    const uint64_t a0 = umma_desc_sw128(smem_u32(T.vt + h * kTcVTile), 2048, 1024);
                    const uint64_t b0 = umma_desc_sw128(smem_u32(T.pt + h * kTcPTile), 16, 1024);
#pragma unroll
                    for (int kk = 0; kk < kTcTokens / 16; ++kk)
                        umma_bf16(tmem + h * 32u + 16u, desc_step(a0, kk * 4096u),
                                  desc_step(b0, (kk / 4) * (kTcN * 128u) + (kk % 4) * 32), idesc_o,
                                  (kk > 0 || !first) ? 1u : 0u);
                    umma_commit(&T.pv_done[h]);
                }
                ++tile;
            }
            if (!ok) {
                report(p.dev_status, PKV_DEV_TIMEOUT);
                *abort_flag = 1;
            }
            // every product issued has retired before the TMEM is released
            umma_commit(T.fin);
            (void)mbar_wait(T.fin, 0);
        }
        __syncwarp();
    } else {
        // ===================== conversion / softmax warpgroup of kv head h =====================
        const int h = warp / 4, wq = warp % 4;        // warpgroup, its warp (TMEM lanes 32 wq ..)
        const int t = threadIdx.x % 128;              // token row of the tile; row d = t of O^T
        const uint32_t bar_id = 1 + h;
        const uint32_t lane_base = tmem + ((uint32_t)(wq * 32) << 16) + h * 32u;
        uint8_t *kt = T.kt + h * kTcKTile, *vt = T.vt + h * kTcVTile, *qt = T.qt + h * kTcQTile,
                *pt = T.pt + h * kTcPTile;
        float *red = T.red + h * 4 * kTcN;
        const float c_lazy = kLazyMax;
        float m[kTcN], lp[kTcN], pp[kTcN], qb[kTcN];
#pragma unroll
        for (int q = 0; q < kTcN; ++q) m[q] = -INFINITY, lp[q] = 0.f, pp[q] = 0.f, qb[q] = 0.f;
        // P' rows of padding query heads stay zero
        for (int i = t; i < (int)(kTcPTile / 16); i += 128)
            *reinterpret_cast<uint4 *>(pt + i * 16) = make_uint4(0, 0, 0, 0);
        uint32_t tile = 0, pieces = 0, phase = 0;
        bool ok = true;
        // this thread's stage of the tile: slot j = t / 16 of the eight, token t % 16
        const int j = t / kStageTokens, tt = t % kStageTokens;
        while (true) {
            // --- stage 0 tells the piece or the stop (every wait is followed by a
            // warpgroup-wide AND, so the warpgroup leaves the loop as one)
            bool w = __all_sync(0xffffffffu, mbar_wait(&L.full_bar[0], phase, abort_flag, p.wait_ns));
            if (!wg_all(bar_id, w)) {
                ok = false;
                break;
            }
            const StageMeta m0 = L.meta[0];
            if (m0.flags & kMetaStop) {
                if (t == 0) {
                    T.info[h] = kTcInfoStop;
                    mbar_arrive(&T.conv_full[h]);
                }
                break;
            }
            const bool first = (m0.flags & kMetaFirst) != 0;
            // own stage; the V and P' tiles are free once the previous tile's
            // product is done; a piece's first tile needs its query rows
            w = __all_sync(0xffffffffu, mbar_wait(&L.full_bar[j], phase, abort_flag, p.wait_ns));
            if (w && tile > 0)
                w = __all_sync(0xffffffffu, mbar_wait(&T.pv_done[h], (tile - 1) & 1, abort_flag, p.wait_ns));
            if (w && first)
                w = __all_sync(0xffffffffu,
                               mbar_wait(&L.qfull_bar[pieces & 1u], (pieces >> 1) & 1u, abort_flag, p.wait_ns));
            if (!wg_all(bar_id, w)) {
                ok = false;
                break;
            }
            const StageMeta mj = L.meta[j];
            const bool have = !(mj.flags & (kMetaPad | kMetaBad));
            const bool valid = have && tt < mj.n_valid;
            const uint8_t *stg = L.stages + (size_t)j * p.stage_bytes;
            float sk = 0.f, sv = 0.f;
            if (first) {
                // the piece's query rows: fp16, K-major, 128-byte swizzle, rows >= G zero;
                // qb = 1152 sum_d q_d of the fp16 rows
                const uint32_t qs = pieces & 1u;
                const __nv_bfloat16 *qrows =
                    reinterpret_cast<const __nv_bfloat16 *>(L.q_slots + qs * p.q_slot_bytes) + (size_t)h * G * D;
                float qpart[2] = {0.f, 0.f};
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    const int c = 2 * t + c2, r = c / 16, ch = c % 16;     // 16-byte chunk ch of row r
                    uint4 w = make_uint4(0, 0, 0, 0);
                    if (r < G) {
                        const uint4 x = *reinterpret_cast<const uint4 *>(qrows + r * D + ch * 8);
                        const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
                        uint32_t ys[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&xs[k]));
                            ys[k] = pack_f16x2(f.x, f.y);
                            const float2 g2 = __half22float2(*reinterpret_cast<const __half2 *>(&ys[k]));
                            qpart[c2] += g2.x + g2.y;
                        }
                        w = make_uint4(ys[0], ys[1], ys[2], ys[3]);
                    }
                    *reinterpret_cast<uint4 *>(qt + (ch / 8) * (kTcN * 128u) + swz(r, ch % 8)) = w;
                }
                // row sums: the 8 threads of a row are consecutive (2 chunks each)
                float rs = qpart[0] + qpart[1];
                rs += __shfl_xor_sync(0xffffffffu, rs, 1);
                rs += __shfl_xor_sync(0xffffffffu, rs, 2);
                rs += __shfl_xor_sync(0xffffffffu, rs, 4);
                if ((t & 7) == 0) red[t / 8] = rs;                      // row r = t / 8 (16 rows)
#pragma unroll
                for (int q = 0; q < kTcN; ++q) m[q] = -INFINITY, lp[q] = 0.f, pp[q] = 0.f;
            }
            // --- this thread's token row: K codes -> fp16 K tile (K-major, swizzled),
            // V codes -> fp16 V tile (MN-major), scales
            if (have) {
                const uint8_t *kc = stg + (size_t)h * kStageTokens * D;
                const uint8_t *vc = kc + p.kv_tile_bytes;
                // this token's scales, read here so that their latency overlaps the
                // conversion (the stages carry only the codes)
                if (valid) {
                    const int64_t srow =
                        (int64_t)(mj.row0 + tt) * p.n_kv_heads + ((int)mj.head_group * kTcHeads + h);
                    sk = __ldg(p.k_scales + srow);
                    sv = __ldg(p.v_scales + srow);
                }
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {              // 16 codes = two 16-byte fp16 chunks
                    const uint4 xk = *reinterpret_cast<const uint4 *>(kc + swz(tt, ch));
                    const uint4 xv = *reinterpret_cast<const uint4 *>(vc + swz(tt, ch));
                    uint4 ka, kb, va_, vb;
                    int8x4_to_biased_half2x2(xk.x, ka.x, ka.y);
                    int8x4_to_biased_half2x2(xk.y, ka.z, ka.w);
                    int8x4_to_biased_half2x2(xk.z, kb.x, kb.y);
                    int8x4_to_biased_half2x2(xk.w, kb.z, kb.w);
                    int8x4_to_biased_half2x2(xv.x, va_.x, va_.y);
                    int8x4_to_biased_half2x2(xv.y, va_.z, va_.w);
                    int8x4_to_biased_half2x2(xv.z, vb.x, vb.y);
                    int8x4_to_biased_half2x2(xv.w, vb.z, vb.w);
                    // d = 16 ch .. 16 ch + 15: fp16 chunks 2 ch and 2 ch + 1
                    const int c0 = 2 * ch, c1 = 2 * ch + 1;
                    *reinterpret_cast<uint4 *>(kt + (c0 / 8) * (kTcTokens * 128u) + swz(t, c0 % 8)) = ka;
                    *reinterpret_cast<uint4 *>(kt + (c1 / 8) * (kTcTokens * 128u) + swz(t, c1 % 8)) = kb;
                    // V tile: 16-token group t / 16 at 4 KiB, panel d / 64 at 2 KiB, 8-token
                    // half at 1 KiB, row t % 8
                    uint8_t *vg = vt + (t / 16) * 4096u + ((t / 8) & 1) * 1024u;
                    *reinterpret_cast<uint4 *>(vg + (c0 / 8) * 2048u + swz(t % 8, c0 % 8)) = va_;
                    *reinterpret_cast<uint4 *>(vg + (c1 / 8) * 2048u + swz(t % 8, c1 % 8)) = vb;
                }
            } else {
                // absent rows: zero V (0 x NaN must not reach O); K rows are masked
                uint8_t *vg = vt + (t / 16) * 4096u + ((t / 8) & 1) * 1024u;
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    *reinterpret_cast<uint4 *>(vg + (c / 8) * 2048u + swz(t % 8, c % 8)) = make_uint4(0, 0, 0, 0);
            }
            // the stage (and at a piece's end the query slot) is converted: hand it back
            const bool last_here = have && (mj.flags & kMetaLast) != 0;
            __syncwarp();
            if (lane == 0) mbar_arrive(&L.empty_bar[j]);
            if (lane == 16) mbar_arrive(&L.empty_bar[j]);
            fence_proxy_async_smem();                 // generic writes -> tensor-core reads
            const bool last = wg_bar_or(bar_id, last_here);
            if (first) {
                // qb from the 16 row sums (written before the barrier)
#pragma unroll
                for (int q = 0; q < kTcN; ++q) qb[q] = kCodeBias * red[q];
            }
            if (t == 0) {
                T.info[h] = first ? kTcInfoFirst : 0u;
                mbar_arrive(&T.conv_full[h]);
            }
            phase ^= 1u;                              // all eight slots consumed once
            // --- softmax over the tile's tokens
            w = __all_sync(0xffffffffu, mbar_wait(&T.s_full[h], tile & 1, abort_flag, p.wait_ns));
            if (!wg_all(bar_id, w)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[kTcN];
            tmem_ld16_async(lane_base, sr);
            tmem_wait_ld();
            float x[kTcN];
            const float c = sk * p.scale_log2;
#pragma unroll
            for (int q = 0; q < kTcN; ++q) x[q] = (valid && q < G) ? (__uint_as_float(sr[q]) - qb[q]) * c : -INFINITY;
            bool up = false;
#pragma unroll
            for (int q = 0; q < kTcN; ++q) up |= x[q] > m[q] + c_lazy;
            if (wg_bar_or(bar_id, up)) {
                // the running maximum moves: the tile's maximum per query head
                float mt[kTcN];
#pragma unroll
                for (int q = 0; q < kTcN; ++q) {
                    float v = x[q];
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
                    mt[q] = v;
                }
                wg_bar(bar_id);                        // red is free (qb was read)
                if (lane == 0)
#pragma unroll
                    for (int q = 0; q < kTcN; ++q) red[wq * kTcN + q] = mt[q];
                wg_bar(bar_id);
                float al[kTcN];
#pragma unroll
                for (int q = 0; q < kTcN; ++q) {
                    const float tm = fmaxf(fmaxf(red[q], red[kTcN + q]), fmaxf(red[2 * kTcN + q], red[3 * kTcN + q]));
                    const float mn = fmaxf(m[q], tm);
                    al[q] = (mn == -INFINITY) ? 1.f : fast_exp2(m[q] - mn);
                    m[q] = mn;
                    lp[q] *= al[q];
                    pp[q] *= al[q];
                }
                if (!first) {
                    // O^T columns of this head hold the piece so far (the previous
                    // tile's product is done): rescale row d = t
                    uint32_t o[kTcN];
                    tmem_ld16_async(lane_base + 16u, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < kTcN; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * al[q]);
                    tmem_st16_async(lane_base + 16u, o);
                    tmem_wait_st();
                }
            }
            // P' = p * v_scale (fp16) into the B tile: row q, token t
            {
                const uint32_t prow = (t / 64) * (kTcN * 128u) + (t % 8) * 2u;
                const uint32_t pch = (t % 64) / 8;
#pragma unroll
                for (int q = 0; q < kTcN; ++q) {
                    const float pr = x[q] == -INFINITY ? 0.f : fast_exp2(x[q] - m[q]);
                    lp[q] += pr;
                    const __half hv = __float2half_rn(pr * sv);
                    pp[q] += __half2float(hv);
                    if (q < G)
                        *reinterpret_cast<__half *>(pt + prow + swz(q, pch)) = hv;
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            wg_bar(bar_id);
            if (t == 0) mbar_arrive(&T.p_full[h]);
            if (last) {
                // --- end of the piece: row sums over the tokens, then O^T row d = t
                w = __all_sync(0xffffffffu, mbar_wait(&T.pv_done[h], tile & 1, abort_flag, p.wait_ns));
                if (!wg_all(bar_id, w)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t o[kTcN];
                tmem_ld16_async(lane_base + 16u, o);
                tmem_wait_ld();
                tc_fence_before();
                float Ls[kTcN], Ps[kTcN];
#pragma unroll
                for (int q = 0; q < kTcN; ++q) {
                    float a = lp[q], b = pp[q];
#pragma unroll
                    for (int off = 16; off >= 1; off >>= 1) {
                        a += __shfl_xor_sync(0xffffffffu, a, off);
                        b += __shfl_xor_sync(0xffffffffu, b, off);
                    }
                    Ls[q] = a;
                    Ps[q] = b;
                }
                if (lane == 0)
#pragma unroll
                    for (int q = 0; q < kTcN; ++q) red[wq * kTcN + q] = Ls[q];
                wg_bar(bar_id);
#pragma unroll
                for (int q = 0; q < kTcN; ++q) Ls[q] = red[q] + red[kTcN + q] + red[2 * kTcN + q] + red[3 * kTcN + q];
                wg_bar(bar_id);
                if (lane == 0)
#pragma unroll
                    for (int q = 0; q < kTcN; ++q) red[wq * kTcN + q] = Ps[q];
                wg_bar(bar_id);
#pragma unroll
                for (int q = 0; q < kTcN; ++q) Ps[q] = red[q] + red[kTcN + q] + red[2 * kTcN + q] + red[3 * kTcN + q];
                // O^T is read out: the next piece's first product may overwrite it
                if (t == 0) mbar_arrive(&T.o_free[h]);
                const int32_t s = m0.seq;
                const int32_t hq0 = (m0.head_group * kTcHeads + h) * G;
                if (m0.flags & kMetaFinal) {
                    __nv_bfloat16 *o_out = p.out + ((int64_t)s * p.n_q_heads + hq0) * D + t;
#pragma unroll
                    for (int q = 0; q < kTcN; ++q)
                        if (q < G)
                            o_out[(size_t)q * D] =
                                __float2bfloat16_rn((__uint_as_float(o[q]) - kCodeBias * Ps[q]) / Ls[q]);
                    if (p.lse_out && t < G) {
                        float mm = 0.f, ll = 1.f;
#pragma unroll
                        for (int q = 0; q < kTcN; ++q)
                            if (q == t) mm = m[q], ll = Ls[q];
                        p.lse_out[(int64_t)s * p.n_q_heads + hq0 + t] = (mm + __log2f(ll)) * 0.69314718055994531f;
                    }
                } else {
                    const int64_t prow = (int64_t)m0.split_index * p.n_q_heads + hq0;
#pragma unroll
                    for (int q = 0; q < kTcN; ++q)
                        if (q < G) p.ws.part_acc[(prow + q) * D + t] = __uint_as_float(o[q]) - kCodeBias * Ps[q];
                    if (t < G) {
                        float mm = 0.f, ll = 1.f;
#pragma unroll
                        for (int q = 0; q < kTcN; ++q)
                            if (q == t) mm = m[q], ll = Ls[q];
                        p.ws.part_ml[prow + t] = make_float2(mm, ll);
                    }
                }
                if (t == 0) mbar_arrive(&L.qempty_bar[pieces & 1u]);
                ++pieces;
            }
            ++tile;
        }
        if (!ok) {
            if (lane == 0) report(p.dev_status, PKV_DEV_TIMEOUT);
            *abort_flag = 1;
        }
    }
    // everyone meets here before the TMEM is released
    tc_fence_before();
    __syncthreads();
    if (warp == kTcIssuerWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols) : "memory");
    }
}

}  // namespace pkv

namespace pkv {

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t decode_workspace_bytes(int32_t n_seqs, int32_t n_q_heads, int32_t head_dim, int64_t capacity)
{
    size_t b = 256;                                                    // header
    b += align_up((size_t)(n_seqs + 1) * sizeof(int32_t), 256);        // seq_prefix
    b += align_up((size_t)n_seqs * sizeof(int2), 256);                 // seg
    b += align_up((size_t)capacity * sizeof(int2), 256);               // items
    b += align_up((size_t)capacity * n_q_heads * sizeof(float2), 256);
    b += align_up((size_t)capacity * n_q_heads * head_dim * sizeof(float), 256);
    return b;
}

bool carve_decode_workspace(void *ws, size_t bytes, int32_t n_seqs, int32_t n_q_heads,
                            int32_t head_dim, DecodeWorkspace *out)
{
    // every array is carved at a multiple of 256 bytes from a 256-byte aligned base
    if (!ws || reinterpret_cast<uintptr_t>(ws) % 256 != 0) return false;
    if (bytes < decode_workspace_bytes(n_seqs, n_q_heads, head_dim, 1)) return false;
    const size_t per = sizeof(int2) + (size_t)n_q_heads * sizeof(float2) +
                       (size_t)n_q_heads * head_dim * sizeof(float);
    int64_t cap = (int64_t)(bytes / per) + 1;
    while (cap > 1 && decode_workspace_bytes(n_seqs, n_q_heads, head_dim, cap) > bytes) --cap;
    if (cap > (int64_t)0x7fffffff) cap = 0x7fffffff;
    uint8_t *p = static_cast<uint8_t *>(ws);
    out->header = reinterpret_cast<uint32_t *>(p);
    p += 256;
    out->seq_prefix = reinterpret_cast<int32_t *>(p);
    p += align_up((size_t)(n_seqs + 1) * sizeof(int32_t), 256);
    out->seg = reinterpret_cast<int2 *>(p);
    p += align_up((size_t)n_seqs * sizeof(int2), 256);
    out->items = reinterpret_cast<int2 *>(p);
    p += align_up((size_t)cap * sizeof(int2), 256);
    out->part_ml = reinterpret_cast<float2 *>(p);
    p += align_up((size_t)cap * n_q_heads * sizeof(float2), 256);
    out->part_acc = reinterpret_cast<float *>(p);
    out->capacity = (int32_t)cap;
    return true;
}

namespace {

// Pool tile map for TMA: preferred is a 3-D view {col, row, head} whose box
// {box_cols, 16, hpc} fetches 16 token rows of hpc heads in one copy; if the
// driver rejects the non-monotonic strides, a {col, head, row} view with one
// box {box_cols, 1, 16} per head.  Returns boxes per column block (1 or hpc),
// or -1 on failure.
int encode_pool_map(CUtensorMap *map, const void *pool, CUtensorMapDataType dt, uint32_t elem_bytes,
                    const pkv_dims &d, int hpc, uint32_t box_cols, CUtensorMapSwizzle swz)
{
    const uint64_t rows = (uint64_t)(d.n_blocks + 1) * d.block_size;
    const uint64_t row_bytes = (uint64_t)d.n_kv_heads * d.head_dim * elem_bytes;
    const uint64_t head_bytes = (uint64_t)d.head_dim * elem_bytes;
    {
        const uint64_t dims[3] = {(uint64_t)d.head_dim, rows, (uint64_t)d.n_kv_heads};
        const uint64_t strides[2] = {row_bytes, head_bytes};
        const uint32_t box[3] = {box_cols, 16u, (uint32_t)hpc};
        if (encode_tensor_map(map, dt, 3, const_cast<void *>(pool), dims, strides, box, swz) ==
            CUDA_SUCCESS)
            return 1;
    }
    const uint64_t dims[3] = {(uint64_t)d.head_dim, (uint64_t)d.n_kv_heads, rows};
    const uint64_t strides[2] = {head_bytes, row_bytes};
    const uint32_t box[3] = {box_cols, 1u, 16u};
    if (encode_tensor_map(map, dt, 3, const_cast<void *>(pool), dims, strides, box, swz) ==
        CUDA_SUCCESS)
        return hpc;
    return -1;
}

// int8 pages of head_dim 128 with up to 8 query heads per kv head (and kv
// heads in multiples of 4) can take the tensor-core kernel; PKV_DECODE_IMPL=tc
// selects it.
bool use_tc_decode(const DecodeArgs &a)
{
    const int G = a.n_q_heads / a.dims.n_kv_heads;
    if (G > kTcMaxGroup || a.dims.n_kv_heads % 4 != 0) return false;
    const char *impl = getenv("PKV_DECODE_IMPL");
    return impl && strcmp(impl, "tc") == 0;
}

// TC: the tensor-core kernel (int8 pages, head_dim 128, G <= 8): two kv
// heads per CTA, one CTA per SM, a ring of exactly one 128-token tile.
template <int D, bool INT8, bool TC = false>
cudaError_t launch_split(const DecodeArgs &a, int num_sms, cudaStream_t stream, const WriteArgs *write)
{
    static_assert(!TC || (INT8 && D == 128), "the tensor-core kernel takes int8 pages of head_dim 128");
    const pkv_dims &d = a.dims;
    const int G = a.n_q_heads / d.n_kv_heads;
    // Launch shape (measured on GB300): one CTA per SM serving up to 8 kv
    // heads; with groups of 8 or more query heads per kv head the consumer
    // warps carry twice the mma work per byte, and 4 kv heads per CTA with two
    // CTAs per SM keep more loads in flight per unit of that work.  int8 pages
    // take 4 kv heads per CTA and two CTAs per SM as well: the consumer warps'
    // in-register code conversion holds ~166 registers, so eight of them fit
    // an SM either way, and two CTAs give two producers and rings (64.6 against
    // 66.1 us on the int8 batch-64 step).
    // (kv heads per CTA: the largest divisor of n_kv_heads up to 8, a multiple
    // of 4 for int8 pages, whose scale rows are copied 16 bytes at a time)
    int hpc = 0, ctas_per_sm = 1;
    for (int c = 8; c >= 1 && hpc == 0; --c)
        if (d.n_kv_heads % c == 0 && (!INT8 || c % 4 == 0)) hpc = c;
    if ((G >= 8 || INT8) && d.n_kv_heads % 4 == 0) {
        hpc = 4;
        ctas_per_sm = 2;
    }
    if (TC) {
        if (G > kTcMaxGroup || d.n_kv_heads % 4 != 0) return cudaErrorInvalidValue;
        hpc = kTcHeads;
        ctas_per_sm = 1;
    }
    if (hpc == 0) return cudaErrorInvalidValue;

    DecodeParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.n_q_heads = a.n_q_heads;
    p.group = G;
    p.hpc = hpc;
    p.n_hg = d.n_kv_heads / hpc;
    p.n_blocks = d.n_blocks;
    p.block_size = d.block_size;
    p.n_kv_heads = d.n_kv_heads;
    p.tables = a.tables;
    p.max_blocks = a.max_blocks;
    p.ctx_lens = a.ctx_lens;
    p.n_seqs = a.n_seqs;
    p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
    p.split_tokens = a.split_tokens;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.lse_out = a.lse_out;
    p.ws = a.ws;
    p.dev_status = a.dev_status;
    p.wait_ns = pipeline_wait_ns();
    p.scale_heads = TC ? 4 : hpc;
    p.tile_stages = TC ? kTcStages : 0;
    p.scales_in_stage = TC ? 0 : 1;
    p.k_scales = a.k_scales;
    p.v_scales = a.v_scales;
    if (!INT8) {
        p.kv_tile_bytes = (uint32_t)(D / 64) * hpc * 16u * 128u;
        p.scale_tile_bytes = 0;
        p.tx_bytes = 2 * p.kv_tile_bytes;
    } else {
        p.kv_tile_bytes = (uint32_t)hpc * 16u * D;
        p.scale_tile_bytes = (uint32_t)p.scale_heads * 16u * 4u;
        p.tx_bytes = 2 * p.kv_tile_bytes + (p.scales_in_stage ? 2 * p.scale_tile_bytes : 0u);
    }
    p.stage_bytes = (uint32_t)align_up(p.tx_bytes, 1024);
    p.q_slot_bytes = (uint32_t)(hpc * G * D * 2);

    CUtensorMap kmap, vmap, ksmap, vsmap;
    memset(&ksmap, 0, sizeof ksmap);
    memset(&vsmap, 0, sizeof vsmap);
    const CUtensorMapDataType dt = INT8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint32_t eb = INT8 ? 1 : 2;
    const uint32_t box_cols = INT8 ? (uint32_t)D : 64u;
    const CUtensorMapSwizzle sw = (INT8 && D == 64) ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
    const int bk = encode_pool_map(&kmap, a.k_pool, dt, eb, d, hpc, box_cols, sw);
    const int bv = encode_pool_map(&vmap, a.v_pool, dt, eb, d, hpc, box_cols, sw);
    if (bk < 0 || bv < 0 || bk != bv) return cudaErrorInvalidValue;
    p.boxes_per_half = bk;
    if (INT8) {
        const uint64_t rows = (uint64_t)(d.n_blocks + 1) * d.block_size;
        const uint64_t dims[2] = {(uint64_t)d.n_kv_heads, rows};
        const uint64_t strides[1] = {(uint64_t)d.n_kv_heads * 4};
        const uint32_t box[2] = {(uint32_t)p.scale_heads, 16u};
        if (encode_tensor_map(&ksmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, (void *)a.k_scales, dims, strides,
                              box, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS ||
            encode_tensor_map(&vsmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, (void *)a.v_scales, dims, strides,
                              box, CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }

    // shared memory: stages fill what one CTA may hold at ctas_per_sm per SM
    const size_t max_smem = 232448;  // 227 KiB per CTA on sm_103
    const size_t per_cta = max_smem / ctas_per_sm - (ctas_per_sm > 1 ? 1024 : 0);
    const size_t fixed = 1024 + 2 * (size_t)p.q_slot_bytes + smem_tail_bytes();
    if (fixed + 2 * (size_t)p.stage_bytes > per_cta) return cudaErrorInvalidValue;
    int stages = (int)((per_cta - fixed) / p.stage_bytes);
    // int8 pages: at most five stages per CTA (measured on GB300: 4, 5 and 6
    // stages of 17 KiB at two CTAs per SM: 64.6, 64.3 and 65.4 us per step)
    const int stage_cap = INT8 ? 5 : kMaxStages;
    stages = stages > stage_cap ? stage_cap : stages;
    size_t smem = fixed + (size_t)stages * p.stage_bytes;
    if (TC) {
        // exactly one tile of stages, then the fp16 tiles from a 1024-byte boundary
        stages = kTcStages;
        smem = 1024 + align_up((size_t)stages * p.stage_bytes + 2 * (size_t)p.q_slot_bytes + smem_tail_bytes(), 1024) +
               tc_smem_extra();
        if (smem > max_smem) return cudaErrorInvalidValue;
    }
    p.n_stages = stages;

    auto kern = TC ? decode_tc_kernel : decode_split_kernel<D, INT8>;
    const int threads = TC ? kTcThreads : 32 * (hpc + 1);
    int occ = 0;
    cudaError_t e = prepare_kernel(reinterpret_cast<const void *>(kern), threads, smem, &occ);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    const int grid = num_sms * (occ < ctas_per_sm ? occ : ctas_per_sm);
    // balanced pieces: about one item per CTA and kv-head group
    const int items_target = (grid + p.n_hg - 1) / p.n_hg;
    const int32_t max_tokens = a.max_blocks * d.block_size;
    // the fused step's write runs in extra CTAs of the plan launch
    int write_mode = 0, write_ctas = 0;
    WriteArgs wa{};
    if (write && write->n_seqs > 0 && write->n_new > 0) {
        wa = *write;
        write_mode = INT8 ? 2 : 1;
        constexpr int64_t warps_per_cta = kPlanThreads / 32;
        const int64_t units = INT8 ? ((int64_t)wa.n_seqs * wa.n_new * 2 * ((d.n_kv_heads + 3) / 4) + warps_per_cta - 1) /
                                         warps_per_cta
                                   : ((int64_t)wa.n_seqs * wa.n_new * (d.n_kv_heads * D / 8) + kPlanThreads - 1) /
                                         kPlanThreads;
        write_ctas = (int)(units < 1 ? 1 : (units > 8 * num_sms ? 8 * num_sms : units));
    }
    // all three launches are programmatic dependents of their predecessor on
    // the stream; each waits (griddepcontrol.wait) before touching memory
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t pc{};
    pc.gridDim = dim3((unsigned)(1 + write_ctas));
    pc.blockDim = dim3(kPlanThreads);
    pc.stream = stream;
    pc.attrs = pdl;
    pc.numAttrs = 1;
    e = cudaLaunchKernelEx(&pc, decode_plan_kernel, a.ctx_lens, a.n_seqs, a.split_tokens, max_tokens, a.n_q_heads,
                           (int32_t)D, d.n_kv_heads, (int32_t)items_target, a.ws, (__nv_bfloat16 *)a.out, a.lse_out,
                           a.dev_status, wa, (int32_t)write_mode, a.write_k_scales, a.write_v_scales);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3((unsigned)grid);
    lc.blockDim = dim3((unsigned)threads);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    lc.attrs = pdl;
    lc.numAttrs = 1;
    e = cudaLaunchKernelEx(&lc, kern, kmap, vmap, ksmap, vsmap, p);
    if (e != cudaSuccess) return e;
    // merge of multi-piece sequences: a warp per (sequence, query head) pair at
    // a time, at most kMergeCtasPerSm CTAs of four warps per SM
    const int64_t warps = (int64_t)a.n_seqs * a.n_q_heads;
    const int64_t merge_ctas = std::min<int64_t>((warps + 3) / 4, (int64_t)num_sms * kMergeCtasPerSm);
    cudaLaunchConfig_t mc{};
    mc.gridDim = dim3((unsigned)std::max<int64_t>(merge_ctas, 1));
    mc.blockDim = dim3(128);   // small CTAs: resident beside the split kernel's before it ends
    mc.stream = stream;
    mc.attrs = pdl;
    mc.numAttrs = 1;
    // fixed splits write partials in proportion to the context (balanced ones
    // about one piece per CTA): only theirs are worth dropping from L2
    return cudaLaunchKernelEx(&mc, decode_merge_kernel<D>, a.ws, a.n_seqs, a.n_q_heads,
                              static_cast<__nv_bfloat16 *>(a.out), a.lse_out, (int32_t)(a.split_tokens > 0));
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, int num_sms, cudaStream_t stream, const WriteArgs *write)
{
    const bool int8 = a.kv_dtype == PKV_KV_INT8;
    if (a.dims.head_dim == 128 && int8 && use_tc_decode(a))
        return launch_split<128, true, true>(a, num_sms, stream, write);
    if (a.dims.head_dim == 128)
        return int8 ? launch_split<128, true>(a, num_sms, stream, write)
                    : launch_split<128, false>(a, num_sms, stream, write);
    return int8 ? launch_split<64, true>(a, num_sms, stream, write) : launch_split<64, false>(a, num_sms, stream, write);
}

}  // namespace pkv
