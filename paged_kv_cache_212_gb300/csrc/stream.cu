// stream.cu -- decode over a host tier streamed through a device scratch pool
// (pagedkv_stream.h): the residency bookkeeping of the scratch pool (least
// recently used slots are reused, slots of the current tile stay pinned), the
// per-tile plan, the staging kernel that reads the host tier straight over the
// CPU-GPU link, and the merge of each tile's attention into a float32 running
// (output, log-sum-exp) state.
#include <math.h>
#include <string.h>

#include <new>
#include <vector>

#include "../../include/pagedkv_stream.h"
#include "common.cuh"
#include "launch.h"

struct pkv_scratch_pool {
    int32_t n_slots = 0, max_seqs = 0;
    // host block -> slot (-1: not resident); grown to the largest id seen (4 bytes
    // per host block, against a host tier of kilobytes per block)
    std::vector<int32_t> slot_of;
    std::vector<int32_t> block_of;                  // slot -> host block (-1: empty)
    // least recently used list over slots: head = next to reuse, tail = newest
    std::vector<int32_t> prev, next;
    int32_t head = -1, tail = -1;
    std::vector<int64_t> pinned_tile;               // tile that last used the slot
    int64_t tiles = 0;
    // two pinned host staging buffers for tile plans, and their copy events
    int32_t *stage[2] = {nullptr, nullptr};
    cudaEvent_t copied[2] = {nullptr, nullptr};
    size_t stage_ints = 0;
    // the copy stream the staging runs on (created at the first streamed call,
    // on the device current then), and the events that order it against the
    // caller's stream: entry (work before the call), staged / decoded per tile parity
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t entry = nullptr, staged[2] = {nullptr, nullptr}, decoded[2] = {nullptr, nullptr};

    void unlink(int32_t s)
    {
        if (prev[s] >= 0) next[prev[s]] = next[s]; else head = next[s];
        if (next[s] >= 0) prev[next[s]] = prev[s]; else tail = prev[s];
        prev[s] = next[s] = -1;
    }
    void push_back(int32_t s)
    {
        prev[s] = tail;
        next[s] = -1;
        if (tail >= 0) next[tail] = s; else head = s;
        tail = s;
    }
    int32_t resident(int32_t hb) const { return hb >= 0 && (size_t)hb < slot_of.size() ? slot_of[hb] : -1; }
    void set_resident(int32_t hb, int32_t slot)
    {
        if ((size_t)hb >= slot_of.size()) slot_of.resize((size_t)hb + 1 + slot_of.size() / 2, -1);
        slot_of[hb] = slot;
    }
    void push_front(int32_t s)
    {
        next[s] = head;
        prev[s] = -1;
        if (head >= 0) prev[head] = s; else tail = s;
        head = s;
    }
};

namespace pkv {

void record_cuda_error(int e);  // api.cu: the value pkv_last_cuda_error() reports

namespace {

constexpr int kPairsAlign = 2;   // pairs start at an even int offset (8-byte int2 loads)

// plan layout in int32 units: tables [n_seqs][width], lens [n_seqs], pairs [cap][2]
// (width = min(cap, max_blocks): a sequence has at most that many blocks in a tile)
size_t pairs_offset(int32_t n_seqs, int32_t width)
{
    const size_t t = (size_t)n_seqs * width + n_seqs;
    return (t + kPairsAlign - 1) / kPairsAlign * kPairsAlign;
}
size_t plan_ints(int32_t n_seqs, int32_t width, int32_t cap) { return pairs_offset(n_seqs, width) + 2 * (size_t)cap; }

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

struct StreamWs {
    void *decode_ws;
    size_t decode_bytes;
    int32_t *plan[2];           // device copies of the tile plans (by tile parity)
    __nv_bfloat16 *tile_out;
    float *tile_lse, *acc, *acc_lse;
};

size_t stream_ws_bytes(int32_t n_seqs, int32_t n_q_heads, int32_t head_dim, int32_t n_slots, int32_t block_size,
                       size_t *decode_bytes)
{
    const size_t d = pkv_decode_workspace_bytes(n_seqs, n_q_heads, head_dim,
                                                (int64_t)n_slots * block_size, 0);
    if (d == 0) return 0;
    if (decode_bytes) *decode_bytes = d;
    const size_t rows = (size_t)n_seqs * n_q_heads;
    return align256(d) + 2 * align256(plan_ints(n_seqs, n_slots, n_slots) * 4) + align256(rows * head_dim * 2) +
           align256(rows * 4) + align256(rows * head_dim * 4) + align256(rows * 4);
}

// Host tier -> scratch pool.  A warp copies one segment of kSegVecs 16-byte
// vectors of the K or the V half of one (host block, slot) pair, all its loads
// issued before its stores; the host tier is read through its device mapping.
// The CPU-GPU link bounds the kernel, so a small grid (two CTAs per SM) keeps
// enough bytes in flight and leaves the SMs to the attention it overlaps.
constexpr int kSegUnroll = 4, kSegVecs = 32 * kSegUnroll;

__global__ void __launch_bounds__(256) stage_blocks_kernel(const uint4 *__restrict__ host_k,
                                                           const uint4 *__restrict__ host_v, uint4 *__restrict__ pool_k,
                                                           uint4 *__restrict__ pool_v, const int2 *__restrict__ pairs,
                                                           int32_t n_host, int32_t n_pool, int64_t block_vecs,
                                                           int64_t segs_per_half, int64_t n_segs, int32_t *dev_status)
{
    const int lane = threadIdx.x & 31;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t seg = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; seg < n_segs; seg += n_warps) {
        const int64_t half = seg / segs_per_half, pr = half >> 1;
        const int64_t off = (seg - half * segs_per_half) * kSegVecs;
        const int2 hs = __ldg(pairs + pr);
        if (hs.x < 0 || hs.x >= n_host || hs.y < 0 || hs.y > n_pool) {
            if (lane == 0 && off == 0 && (half & 1) == 0) report(dev_status, PKV_DEV_BAD_BLOCK_ID);
            continue;
        }
        const uint4 *src = ((half & 1) ? host_v : host_k) + (int64_t)hs.x * block_vecs + off;
        uint4 *dst = ((half & 1) ? pool_v : pool_k) + (int64_t)hs.y * block_vecs + off;
        const int64_t left = block_vecs - off;
        uint4 x[kSegUnroll];
#pragma unroll
        for (int u = 0; u < kSegUnroll; ++u)
            if (u * 32 + lane < left) x[u] = src[u * 32 + lane];
#pragma unroll
        for (int u = 0; u < kSegUnroll; ++u)
            if (u * 32 + lane < left) dst[u * 32 + lane] = x[u];
    }
}

// One warp per (sequence, query head) row: the tile's normalised output o_t and
// log-sum-exp lse_t merge into the running (acc, lse) -- acc stays normalised:
// acc = (acc e^(lse - M) + o_t e^(lse_t - M)) / (e^(lse - M) + e^(lse_t - M)).
template <int D>
__global__ void __launch_bounds__(256) merge_tile_kernel(const __nv_bfloat16 *__restrict__ tile_out,
                                                         const float *__restrict__ tile_lse, float *__restrict__ acc,
                                                         float *__restrict__ acc_lse, int64_t n_rows, int first)
{
    constexpr int EPL = D / 32;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= n_rows) return;
    const float lt = tile_lse[row];
    const __nv_bfloat16 *o = tile_out + row * D + lane * EPL;
    float *a = acc + row * D + lane * EPL;
    float ot[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) ot[e] = __bfloat162float(o[e]);
    if (first) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) a[e] = ot[e];
        if (lane == 0) acc_lse[row] = lt;
        return;
    }
    const float la = acc_lse[row];
    const float M = fmaxf(la, lt);
    if (M == -INFINITY) return;   // neither has any token yet
    const float wa = expf(la - M), wt = expf(lt - M);
    const float inv = 1.f / (wa + wt);
#pragma unroll
    for (int e = 0; e < EPL; ++e) a[e] = (a[e] * wa + ot[e] * wt) * inv;
    __syncwarp();
    if (lane == 0) acc_lse[row] = M + logf(wa + wt);
}

template <int D>
__global__ void __launch_bounds__(256) finalize_tiles_kernel(const float *__restrict__ acc,
                                                             const float *__restrict__ acc_lse,
                                                             __nv_bfloat16 *__restrict__ out, float *__restrict__ lse_out,
                                                             int64_t n_rows)
{
    constexpr int EPL = D / 32;
    const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= n_rows) return;
    const float *a = acc + row * D + lane * EPL;
    __nv_bfloat16 *o = out + row * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; e += 2) *reinterpret_cast<uint32_t *>(o + e) = pack_bf16x2(a[e], a[e + 1]);
    if (lse_out && lane == 0) lse_out[row] = acc_lse[row];
}

int cuda_err(cudaError_t e)
{
    if (e == cudaSuccess) return PKV_OK;
    record_cuda_error((int)e);
    return PKV_ERR_CUDA;
}

// device pointer of pinned, mapped host memory (PKV_ERR_INVALID_ARG otherwise)
int mapped(const void *host, const void **dev)
{
    void *d = nullptr;
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, host) != cudaSuccess) {
        (void)cudaGetLastError();
        return PKV_ERR_INVALID_ARG;
    }
    if (at.type != cudaMemoryTypeHost) return PKV_ERR_INVALID_ARG;
    if (cudaHostGetDevicePointer(&d, const_cast<void *>(host), 0) != cudaSuccess || !d) {
        (void)cudaGetLastError();
        return PKV_ERR_INVALID_ARG;
    }
    *dev = d;
    return PKV_OK;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

int pkv_sp_create(int32_t n_slots, int32_t max_seqs, pkv_scratch_pool **out)
{
    if (!out || n_slots <= 0 || max_seqs <= 0) return PKV_ERR_INVALID_ARG;
    pkv_scratch_pool *sp = new (std::nothrow) pkv_scratch_pool();
    if (!sp) return PKV_ERR_INVALID_ARG;
    sp->n_slots = n_slots;
    sp->max_seqs = max_seqs;
    sp->block_of.assign(n_slots, -1);
    sp->prev.assign(n_slots, -1);
    sp->next.assign(n_slots, -1);
    sp->pinned_tile.assign(n_slots, -1);
    for (int32_t s = 0; s < n_slots; ++s) sp->push_back(s);   // slot 0 is reused first
    sp->stage_ints = plan_ints(max_seqs, n_slots, n_slots);
    *out = sp;
    return PKV_OK;
}

void pkv_sp_destroy(pkv_scratch_pool *sp)
{
    if (!sp) return;
    if (sp->copy_stream) (void)cudaStreamSynchronize(sp->copy_stream);
    for (int b = 0; b < 2; ++b) {
        if (sp->copied[b]) {
            (void)cudaEventSynchronize(sp->copied[b]);
            (void)cudaEventDestroy(sp->copied[b]);
        }
        if (sp->staged[b]) (void)cudaEventDestroy(sp->staged[b]);
        if (sp->decoded[b]) {
            (void)cudaEventSynchronize(sp->decoded[b]);
            (void)cudaEventDestroy(sp->decoded[b]);
        }
        if (sp->stage[b]) (void)cudaFreeHost(sp->stage[b]);
    }
    if (sp->entry) (void)cudaEventDestroy(sp->entry);
    if (sp->copy_stream) (void)cudaStreamDestroy(sp->copy_stream);
    delete sp;
}

int32_t pkv_sp_lookup(const pkv_scratch_pool *sp, int32_t host_block)
{
    return sp ? sp->resident(host_block) : -1;
}

int pkv_sp_invalidate(pkv_scratch_pool *sp, int32_t host_block)
{
    if (!sp) return PKV_ERR_INVALID_ARG;
    const int32_t s = sp->resident(host_block);
    if (s < 0) return PKV_OK;
    sp->slot_of[host_block] = -1;
    sp->block_of[s] = -1;
    sp->unlink(s);
    sp->push_front(s);   // an empty slot is reused first
    return PKV_OK;
}

int pkv_sp_plan_tile(pkv_scratch_pool *sp, const int32_t *host_tables, int32_t max_blocks, const int32_t *ctx_lens,
                     int32_t n_seqs, int32_t block_size, int32_t tile_blocks, int32_t *cursor, int32_t *tile_tables,
                     int32_t *tile_lens, int32_t *pairs, int32_t *n_pairs, int32_t *done)
{
    if (!sp || !cursor || !tile_tables || !tile_lens || !pairs || !n_pairs || !done || n_seqs < 0 ||
        n_seqs > sp->max_seqs || block_size <= 0 || max_blocks <= 0 || (n_seqs > 0 && (!host_tables || !ctx_lens)))
        return PKV_ERR_INVALID_ARG;
    for (int32_t s = 0; s < n_seqs; ++s)
        if (ctx_lens[s] < 0 || (int64_t)ctx_lens[s] > (int64_t)max_blocks * block_size) return PKV_ERR_OUT_OF_RANGE;
    const int32_t n_slots = sp->n_slots;
    const int32_t cap = tile_blocks <= 0 || tile_blocks > n_slots ? n_slots : tile_blocks;
    const int32_t width = cap < max_blocks ? cap : max_blocks;
    auto blocks_of = [&](int32_t q) { return (ctx_lens[q] + block_size - 1) / block_size; };
    // the tile's host ids are checked before any state changes
    {
        int32_t s = cursor[0], j = cursor[1], taken = 0;
        if (s < 0 || j < 0) return PKV_ERR_INVALID_ARG;
        while (s < n_seqs && taken < cap) {
            if (j >= blocks_of(s)) {
                ++s;
                j = 0;
                continue;
            }
            if (host_tables[(int64_t)s * max_blocks + j] < 0) return PKV_ERR_OUT_OF_RANGE;
            ++j;
            ++taken;
        }
    }
    for (int64_t i = 0; i < (int64_t)n_seqs * width; ++i) tile_tables[i] = n_slots;   // the scratch slot
    for (int32_t s = 0; s < n_seqs; ++s) tile_lens[s] = 0;
    std::vector<int32_t> used(n_seqs, 0);
    const int64_t tile = ++sp->tiles;
    int32_t s = cursor[0], j = cursor[1], taken = 0, np = 0;
    while (s < n_seqs && taken < cap) {
        if (j >= blocks_of(s)) {
            ++s;
            j = 0;
            continue;
        }
        const int32_t hb = host_tables[(int64_t)s * max_blocks + j];
        int32_t slot = sp->resident(hb);
        if (slot < 0) {
            slot = sp->head;   // least recently used; every slot of this tile sits behind it
            if (sp->pinned_tile[slot] == tile) return PKV_ERR_STATE;   // cannot happen: taken < n_slots
            if (sp->block_of[slot] >= 0) sp->slot_of[sp->block_of[slot]] = -1;
            sp->block_of[slot] = hb;
            sp->set_resident(hb, slot);
            pairs[2 * np] = hb;
            pairs[2 * np + 1] = slot;
            ++np;
        }
        sp->pinned_tile[slot] = tile;
        sp->unlink(slot);
        sp->push_back(slot);
        tile_tables[(int64_t)s * width + used[s]++] = slot;
        tile_lens[s] += (int32_t)((int64_t)ctx_lens[s] - (int64_t)j * block_size < block_size
                                      ? ctx_lens[s] - j * block_size : block_size);
        ++j;
        ++taken;
    }
    while (s < n_seqs && j >= blocks_of(s)) {
        ++s;
        j = 0;
    }
    cursor[0] = s;
    cursor[1] = j;
    *n_pairs = np;
    *done = s >= n_seqs ? 1 : 0;
    return PKV_OK;
}

int paged_kv_stage_blocks(const int32_t *pairs, int32_t n_pairs, const pkv_bf16 *host_k, const pkv_bf16 *host_v,
                          int32_t n_host_blocks, pkv_bf16 *pool_k, pkv_bf16 *pool_v, pkv_dims pool_dims,
                          int32_t *dev_status, pkv_stream_t stream)
{
    if (n_pairs < 0 || n_host_blocks < 0 || pool_dims.n_blocks < 0 || pool_dims.block_size <= 0 ||
        pool_dims.n_kv_heads <= 0)
        return PKV_ERR_INVALID_ARG;
    if (pool_dims.head_dim != 64 && pool_dims.head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (n_pairs == 0) return PKV_OK;
    if (!pairs || !host_k || !host_v || !pool_k || !pool_v || (reinterpret_cast<uintptr_t>(pairs) & 7) != 0 ||
        (reinterpret_cast<uintptr_t>(pool_k) & 15) != 0 || (reinterpret_cast<uintptr_t>(pool_v) & 15) != 0 ||
        (reinterpret_cast<uintptr_t>(host_k) & 15) != 0 || (reinterpret_cast<uintptr_t>(host_v) & 15) != 0)
        return PKV_ERR_INVALID_ARG;
    const void *dk = nullptr, *dv = nullptr;
    int st = mapped(host_k, &dk);
    if (st == PKV_OK) st = mapped(host_v, &dv);
    if (st != PKV_OK) return st;
    const int64_t block_vecs = (int64_t)pool_dims.block_size * pool_dims.n_kv_heads * pool_dims.head_dim * 2 / 16;
    const int64_t segs_per_half = (block_vecs + kSegVecs - 1) / kSegVecs;
    const int64_t n_segs = (int64_t)n_pairs * 2 * segs_per_half;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cuda_err(cudaGetLastError());
    int64_t grid = (n_segs + 7) / 8;
    if (grid > 2 * (int64_t)sms) grid = 2 * (int64_t)sms;
    stage_blocks_kernel<<<(unsigned)grid, 256, 0, (cudaStream_t)stream>>>(
        (const uint4 *)dk, (const uint4 *)dv, (uint4 *)pool_k, (uint4 *)pool_v, (const int2 *)pairs, n_host_blocks,
        pool_dims.n_blocks, block_vecs, segs_per_half, n_segs, dev_status);
    return cuda_err(cudaGetLastError());
}

size_t pkv_streamed_workspace_bytes(int32_t n_seqs, int32_t n_q_heads, int32_t head_dim, int32_t n_slots,
                                    int32_t block_size)
{
    if (n_seqs <= 0 || n_q_heads <= 0 || (head_dim != 64 && head_dim != 128) || n_slots <= 0 || block_size <= 0)
        return 0;
    return stream_ws_bytes(n_seqs, n_q_heads, head_dim, n_slots, block_size, nullptr);
}

int paged_decode_streamed(const pkv_bf16 *q, int32_t n_q_heads, const pkv_bf16 *host_k, const pkv_bf16 *host_v,
                          int32_t n_host_blocks, pkv_bf16 *pool_k, pkv_bf16 *pool_v, pkv_dims pool_dims,
                          pkv_scratch_pool *sp, const int32_t *host_tables, int32_t max_blocks,
                          const int32_t *ctx_lens, int32_t n_seqs, float softmax_scale, pkv_bf16 *out,
                          float *lse_out, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                          pkv_stream_t stream)
{
    if (!sp || n_seqs < 0 || n_q_heads <= 0 || n_host_blocks < 0 || max_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (n_seqs == 0) return PKV_OK;
    if (pool_dims.n_blocks != sp->n_slots || n_seqs > sp->max_seqs) return PKV_ERR_INVALID_ARG;
    if (!q || !out || !host_tables || !ctx_lens || !workspace) return PKV_ERR_INVALID_ARG;
    if (!(softmax_scale > 0.f) || !isfinite(softmax_scale)) return PKV_ERR_INVALID_ARG;   // as the decode itself
    const int32_t D = pool_dims.head_dim, bs = pool_dims.block_size, n_slots = sp->n_slots;
    if (D != 64 && D != 128) return PKV_ERR_UNSUPPORTED;
    for (int64_t i = 0; i < (int64_t)n_seqs; ++i) {
        if (ctx_lens[i] < 0 || (int64_t)ctx_lens[i] > (int64_t)max_blocks * bs) return PKV_ERR_OUT_OF_RANGE;
        for (int32_t j = 0; j < (ctx_lens[i] + bs - 1) / bs; ++j) {
            const int32_t hb = host_tables[i * max_blocks + j];
            if (hb < 0 || hb >= n_host_blocks) return PKV_ERR_OUT_OF_RANGE;
        }
    }
    size_t decode_bytes = 0;
    const size_t need = stream_ws_bytes(n_seqs, n_q_heads, D, n_slots, bs, &decode_bytes);
    if (need == 0) return PKV_ERR_INVALID_ARG;
    if (workspace_bytes < need || reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return PKV_ERR_WORKSPACE;
    // check the host tier's device mapping once (staging would fail per tile)
    const void *dk = nullptr, *dv = nullptr;
    int st = mapped(host_k, &dk);
    if (st == PKV_OK) st = mapped(host_v, &dv);
    if (st != PKV_OK) return st;
    // lazily: pinned staging buffers, the copy stream and the events
    for (int b = 0; b < 2; ++b) {
        if (!sp->stage[b]) {
            void *p = nullptr;
            if (cudaHostAlloc(&p, sp->stage_ints * 4, cudaHostAllocDefault) != cudaSuccess) return PKV_ERR_CUDA;
            sp->stage[b] = static_cast<int32_t *>(p);
        }
        for (cudaEvent_t *e : {&sp->copied[b], &sp->staged[b], &sp->decoded[b]})
            if (!*e && cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return PKV_ERR_CUDA;
    }
    if (!sp->entry && cudaEventCreateWithFlags(&sp->entry, cudaEventDisableTiming) != cudaSuccess) return PKV_ERR_CUDA;
    if (!sp->copy_stream && cudaStreamCreateWithFlags(&sp->copy_stream, cudaStreamNonBlocking) != cudaSuccess)
        return PKV_ERR_CUDA;
    uint8_t *w = static_cast<uint8_t *>(workspace);
    StreamWs ws;
    ws.decode_ws = w;
    ws.decode_bytes = decode_bytes;
    w += align256(decode_bytes);
    for (int b = 0; b < 2; ++b) {
        ws.plan[b] = reinterpret_cast<int32_t *>(w);
        w += align256(plan_ints(n_seqs, n_slots, n_slots) * 4);
    }
    const size_t rows = (size_t)n_seqs * n_q_heads;
    ws.tile_out = reinterpret_cast<__nv_bfloat16 *>(w);
    w += align256(rows * D * 2);
    ws.tile_lse = reinterpret_cast<float *>(w);
    w += align256(rows * 4);
    ws.acc = reinterpret_cast<float *>(w);
    w += align256(rows * D * 4);
    ws.acc_lse = reinterpret_cast<float *>(w);

    // Tiles of at most n_slots / 2 blocks when the batch does not fit the pool:
    // the least recently used slots a tile stages into are then never those
    // of the tile before it, so the staging of tile t + 1 (copy stream) only
    // waits for the attention of tile t - 1 and overlaps that of tile t.
    int64_t total_blocks = 0;
    for (int32_t i = 0; i < n_seqs; ++i) total_blocks += (ctx_lens[i] + bs - 1) / bs;
    const bool overlap = total_blocks > n_slots && n_slots >= 2;
    const int32_t tile_blocks = overlap ? n_slots / 2 : n_slots;
    cudaStream_t s = (cudaStream_t)stream, c = sp->copy_stream;
    if (cudaEventRecord(sp->entry, s) != cudaSuccess || cudaStreamWaitEvent(c, sp->entry, 0) != cudaSuccess)
        return cuda_err(cudaGetLastError());
    const int32_t width = tile_blocks < max_blocks ? tile_blocks : max_blocks;   // tile table row length
    const size_t lens_off = (size_t)n_seqs * width, pairs_off = pairs_offset(n_seqs, width);
    const size_t pints = plan_ints(n_seqs, width, tile_blocks);
    int32_t cursor[2] = {0, 0}, done = 0;
    int first = 1;
    for (int64_t t = 0; !done; ++t) {
        const int b = (int)(t & 1);
        if (cudaEventSynchronize(sp->copied[b]) != cudaSuccess) return cuda_err(cudaGetLastError());   // tile t - 2's copy read it
        int32_t *plan = sp->stage[b];
        int32_t np = 0;
        st = pkv_sp_plan_tile(sp, host_tables, max_blocks, ctx_lens, n_seqs, bs, tile_blocks, cursor, plan,
                              plan + lens_off, plan + pairs_off, &np, &done);
        if (st != PKV_OK) return st;
        // copy stream: wait until no earlier tile still reads the slots (and the
        // device plan buffer) this tile overwrites, then plan copy and staging
        const int64_t need = overlap ? t - 2 : t - 1;
        if (need >= 0 && cudaStreamWaitEvent(c, sp->decoded[need & 1], 0) != cudaSuccess)
            return cuda_err(cudaGetLastError());
        if (cudaMemcpyAsync(ws.plan[b], plan, pints * 4, cudaMemcpyHostToDevice, c) != cudaSuccess ||
            cudaEventRecord(sp->copied[b], c) != cudaSuccess)
            return cuda_err(cudaGetLastError());
        st = paged_kv_stage_blocks(ws.plan[b] + pairs_off, np, host_k, host_v, n_host_blocks, pool_k, pool_v,
                                   pool_dims, dev_status, c);
        if (st != PKV_OK) return st;
        if (cudaEventRecord(sp->staged[b], c) != cudaSuccess || cudaStreamWaitEvent(s, sp->staged[b], 0) != cudaSuccess)
            return cuda_err(cudaGetLastError());
        // caller's stream: attention over the tile, then its merge into the running
        // state (a batch in one tile is attended straight into out and lse_out)
        const bool only = first && done;
        st = paged_decode_attention(q, n_q_heads, pool_k, pool_v, nullptr, nullptr, PKV_KV_BF16, pool_dims, ws.plan[b],
                                    width, ws.plan[b] + lens_off, n_seqs, softmax_scale, 0,
                                    only ? out : reinterpret_cast<pkv_bf16 *>(ws.tile_out),
                                    only ? lse_out : ws.tile_lse, ws.decode_ws, ws.decode_bytes, dev_status, stream);
        if (st != PKV_OK) return st;
        if (cudaEventRecord(sp->decoded[b], s) != cudaSuccess) return cuda_err(cudaGetLastError());
        if (only) return PKV_OK;
        const unsigned grid = (unsigned)((rows + 7) / 8);
        if (D == 128)
            merge_tile_kernel<128><<<grid, 256, 0, s>>>(ws.tile_out, ws.tile_lse, ws.acc, ws.acc_lse, (int64_t)rows, first);
        else
            merge_tile_kernel<64><<<grid, 256, 0, s>>>(ws.tile_out, ws.tile_lse, ws.acc, ws.acc_lse, (int64_t)rows, first);
        if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
        first = 0;
    }
    const unsigned grid = (unsigned)((rows + 7) / 8);
    if (D == 128)
        finalize_tiles_kernel<128><<<grid, 256, 0, s>>>(ws.acc, ws.acc_lse, (__nv_bfloat16 *)out, lse_out, (int64_t)rows);
    else
        finalize_tiles_kernel<64><<<grid, 256, 0, s>>>(ws.acc, ws.acc_lse, (__nv_bfloat16 *)out, lse_out, (int64_t)rows);
    return cuda_err(cudaGetLastError());
}

}  // extern "C"
