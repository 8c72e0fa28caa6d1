// block_manager.cpp -- host-side block manager behind pagedkv_blocks.h: the
// free stack and reference counts of a block pool, and the per-slot tables,
// lengths and admission order a continuous-batching engine keeps.  Every call
// checks its whole request before changing anything, so a failing call leaves
// the manager as it was.
#include <stdint.h>

#include <algorithm>
#include <new>
#include <vector>

#include "../../include/pagedkv_blocks.h"

struct pkv_block_manager {
    int32_t n_blocks, block_size, n_slots, max_blocks;
    std::vector<int32_t> free_stack;   // top = back(): the next block handed out
    std::vector<int32_t> refs;         // per block; 0 = free
    int32_t peak_used = 0;
    std::vector<std::vector<int32_t>> tables;
    std::vector<int32_t> lens;
    std::vector<uint8_t> active;
    std::vector<int64_t> admit_no;     // admission order (larger = newer)
    int64_t admits = 0;

    int32_t used() const { return n_blocks - (int32_t)free_stack.size(); }
    int32_t pop()
    {
        const int32_t b = free_stack.back();
        free_stack.pop_back();
        refs[b] = 1;
        peak_used = std::max(peak_used, used());
        return b;
    }
    void drop(int32_t b)
    {
        if (--refs[b] == 0) free_stack.push_back(b);
    }
    bool valid_slot(int32_t s) const { return s >= 0 && s < n_slots; }
    // blocks the coming step needs for slot s: one if its table is full (the
    // token at position len starts a new block), one if the block holding
    // position len is shared (copy-on-write), else none
    int32_t step_need(int32_t s) const
    {
        const std::vector<int32_t> &t = tables[s];
        if ((int64_t)t.size() * block_size <= lens[s]) return 1;
        return refs[t[lens[s] / block_size]] > 1 ? 1 : 0;
    }
    int32_t total_need() const
    {
        int32_t n = 0;
        for (int32_t s = 0; s < n_slots; ++s)
            if (active[s]) n += step_need(s);
        return n;
    }
    void release(int32_t s)
    {
        for (int32_t b : tables[s]) drop(b);
        tables[s].clear();
        lens[s] = 0;
        active[s] = 0;
    }
};

extern "C" {

int pkv_bm_create(int32_t n_blocks, int32_t block_size, int32_t n_slots, int32_t max_blocks,
                  pkv_block_manager **out)
{
    if (!out || n_blocks <= 0 || block_size <= 0 || n_slots <= 0 || max_blocks <= 0) return PKV_ERR_INVALID_ARG;
    pkv_block_manager *bm = new (std::nothrow) pkv_block_manager();
    if (!bm) return PKV_ERR_INVALID_ARG;
    bm->n_blocks = n_blocks;
    bm->block_size = block_size;
    bm->n_slots = n_slots;
    bm->max_blocks = max_blocks;
    bm->free_stack.resize(n_blocks);
    for (int32_t i = 0; i < n_blocks; ++i) bm->free_stack[i] = n_blocks - 1 - i;   // block 0 on top
    bm->refs.assign(n_blocks, 0);
    bm->tables.assign(n_slots, {});
    bm->lens.assign(n_slots, 0);
    bm->active.assign(n_slots, 0);
    bm->admit_no.assign(n_slots, 0);
    *out = bm;
    return PKV_OK;
}

void pkv_bm_destroy(pkv_block_manager *bm) { delete bm; }

int pkv_bm_alloc(pkv_block_manager *bm, int32_t *block)
{
    if (!bm || !block) return PKV_ERR_INVALID_ARG;
    if (bm->free_stack.empty()) return PKV_ERR_OUT_OF_BLOCKS;
    *block = bm->pop();
    return PKV_OK;
}

int pkv_bm_free(pkv_block_manager *bm, const int32_t *blocks, int32_t n)
{
    if (!bm || n < 0 || (n > 0 && !blocks)) return PKV_ERR_INVALID_ARG;
    // references dropped per block must not exceed those held
    std::vector<int32_t> take;
    take.reserve(n);
    for (int32_t i = 0; i < n; ++i) {
        const int32_t b = blocks[i];
        if (b < 0 || b >= bm->n_blocks) return PKV_ERR_INVALID_ARG;
        take.push_back(b);
    }
    std::vector<int32_t> sorted(take);
    std::sort(sorted.begin(), sorted.end());
    for (size_t i = 0; i < sorted.size();) {
        size_t j = i;
        while (j < sorted.size() && sorted[j] == sorted[i]) ++j;
        if ((int64_t)(j - i) > bm->refs[sorted[i]]) return PKV_ERR_STATE;
        i = j;
    }
    for (int32_t b : take) bm->drop(b);
    return PKV_OK;
}

int32_t pkv_bm_num_free(const pkv_block_manager *bm) { return bm ? (int32_t)bm->free_stack.size() : 0; }

int32_t pkv_bm_peak_used(const pkv_block_manager *bm) { return bm ? bm->peak_used : 0; }

int32_t pkv_bm_refcount(const pkv_block_manager *bm, int32_t block)
{
    if (!bm || block < 0 || block >= bm->n_blocks) return -1;
    return bm->refs[block];
}

int pkv_bm_can_admit(const pkv_block_manager *bm, const int32_t *lengths, int32_t n, int32_t *ok)
{
    if (!bm || !ok || n < 0 || (n > 0 && !lengths)) return PKV_ERR_INVALID_ARG;
    int64_t need = 0;
    for (int32_t i = 0; i < n; ++i) {
        if (lengths[i] < 0) return PKV_ERR_INVALID_ARG;
        need += ((int64_t)lengths[i] + 1 + bm->block_size - 1) / bm->block_size;
    }
    *ok = need <= (int64_t)bm->free_stack.size() ? 1 : 0;
    return PKV_OK;
}

int pkv_bm_admit(pkv_block_manager *bm, int32_t slot, int32_t n_tokens)
{
    if (!bm || !bm->valid_slot(slot) || n_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (bm->active[slot]) return PKV_ERR_STATE;
    if ((int64_t)n_tokens >= (int64_t)bm->max_blocks * bm->block_size) return PKV_ERR_OUT_OF_RANGE;
    const int32_t nb = (n_tokens + bm->block_size - 1) / bm->block_size;
    if (nb > (int32_t)bm->free_stack.size()) return PKV_ERR_OUT_OF_BLOCKS;
    std::vector<int32_t> &t = bm->tables[slot];
    t.clear();
    for (int32_t i = 0; i < nb; ++i) t.push_back(bm->pop());
    bm->lens[slot] = n_tokens;
    bm->active[slot] = 1;
    bm->admit_no[slot] = ++bm->admits;
    return PKV_OK;
}

int pkv_bm_release(pkv_block_manager *bm, int32_t slot)
{
    if (!bm || !bm->valid_slot(slot)) return PKV_ERR_INVALID_ARG;
    bm->release(slot);
    return PKV_OK;
}

int pkv_bm_fork(pkv_block_manager *bm, int32_t src_slot, int32_t dst_slot)
{
    if (!bm || !bm->valid_slot(src_slot) || !bm->valid_slot(dst_slot) || src_slot == dst_slot)
        return PKV_ERR_INVALID_ARG;
    if (!bm->active[src_slot] || bm->active[dst_slot]) return PKV_ERR_STATE;
    bm->tables[dst_slot] = bm->tables[src_slot];
    for (int32_t b : bm->tables[dst_slot]) ++bm->refs[b];
    bm->lens[dst_slot] = bm->lens[src_slot];
    bm->active[dst_slot] = 1;
    bm->admit_no[dst_slot] = ++bm->admits;
    return PKV_OK;
}

int pkv_bm_reserve_step(pkv_block_manager *bm, int32_t *victims, int32_t *n_victims)
{
    if (!bm || !victims || !n_victims) return PKV_ERR_INVALID_ARG;
    int32_t nv = 0;
    while (true) {
        int32_t newest = -1;
        for (int32_t s = 0; s < bm->n_slots; ++s)
            if (bm->active[s] && (newest < 0 || bm->admit_no[s] > bm->admit_no[newest])) newest = s;
        if (newest < 0 || bm->total_need() <= (int32_t)bm->free_stack.size()) break;
        bm->release(newest);
        victims[nv++] = newest;
    }
    *n_victims = nv;
    return PKV_OK;
}

int pkv_bm_begin_step(pkv_block_manager *bm, int32_t *copies, int32_t *n_copies)
{
    if (!bm || !copies || !n_copies) return PKV_ERR_INVALID_ARG;
    for (int32_t s = 0; s < bm->n_slots; ++s)
        if (bm->active[s] && (int64_t)bm->lens[s] >= (int64_t)bm->max_blocks * bm->block_size)
            return PKV_ERR_OUT_OF_RANGE;
    if (bm->total_need() > (int32_t)bm->free_stack.size()) return PKV_ERR_OUT_OF_BLOCKS;
    int32_t nc = 0;
    for (int32_t s = 0; s < bm->n_slots; ++s) {
        if (!bm->active[s]) continue;
        std::vector<int32_t> &t = bm->tables[s];
        if ((int64_t)t.size() * bm->block_size <= bm->lens[s]) {
            t.push_back(bm->pop());
        } else {
            const int32_t j = bm->lens[s] / bm->block_size;
            const int32_t old = t[j];
            if (bm->refs[old] > 1) {
                const int32_t fresh = bm->pop();
                --bm->refs[old];   // still held by the other sharers
                t[j] = fresh;
                copies[2 * nc] = old;
                copies[2 * nc + 1] = fresh;
                ++nc;
            }
        }
    }
    *n_copies = nc;
    return PKV_OK;
}

int pkv_bm_end_step(pkv_block_manager *bm)
{
    if (!bm) return PKV_ERR_INVALID_ARG;
    for (int32_t s = 0; s < bm->n_slots; ++s)
        if (bm->active[s]) ++bm->lens[s];
    return PKV_OK;
}

int pkv_bm_export(const pkv_block_manager *bm, int32_t *tables, int32_t *lens, int32_t *active)
{
    if (!bm) return PKV_ERR_INVALID_ARG;
    for (int32_t s = 0; s < bm->n_slots; ++s) {
        if (tables) {
            int32_t *row = tables + (int64_t)s * bm->max_blocks;
            const std::vector<int32_t> &t = bm->tables[s];
            for (int32_t j = 0; j < bm->max_blocks; ++j)
                row[j] = j < (int32_t)t.size() ? t[j] : bm->n_blocks;
        }
        if (lens) lens[s] = bm->active[s] ? bm->lens[s] : 0;
        if (active) active[s] = bm->active[s];
    }
    return PKV_OK;
}

}  // extern "C"
