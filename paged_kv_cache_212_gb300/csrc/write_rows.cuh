// write_rows.cuh -- the page-write work (bf16 copy and int8 quantisation) as
// device functions over a flat index space, shared by the stand-alone write
// kernels and by the fused decode step, which runs the write in the same launch
// as its plan.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace pkv {

// Pool row of token t of the sequence whose table row is `table_row`, or -1
// (and a status bit) when the block is outside the table or the id outside
// [0, n_blocks].  tiny-llm paged_kv.py, module docstring: token t lives at
// (table[t // block_size], t % block_size).
__device__ __forceinline__ int64_t pool_row_of(const int32_t *table_row, int32_t max_blocks,
                                               int32_t n_blocks, int32_t block_size, int64_t t,
                                               int32_t *dev_status)
{
    if (t < 0 || t >= (int64_t)max_blocks * block_size) {
        report(dev_status, PKV_DEV_BAD_POSITION);
        return -1;
    }
    // 0 <= t < 2^32 (an int32 start position plus an int32 row index): 32-bit division
    const uint32_t tt = (uint32_t)t, blk = tt / (uint32_t)block_size;
    const int32_t b = __ldg(table_row + blk);
    if (b < 0 || b > n_blocks) {
        report(dev_status, PKV_DEV_BAD_BLOCK_ID);
        return -1;
    }
    return (int64_t)b * block_size + (tt - blk * (uint32_t)block_size);
}

// x / d for a non-negative flat index x and a positive d, in 32 bits when the
// whole index space is below 2^31 (narrow, the same for every thread), else
// in 64.
__device__ __forceinline__ int64_t index_div(int64_t x, int32_t d, bool narrow)
{
    return narrow ? (int64_t)((uint32_t)x / (uint32_t)d) : x / d;
}

// Native bf16 write: 16-byte vector i of the [n_seqs * n_new rows][Hkv * D]
// new K and V rows goes to the same vector of its token's pool row.  Threads
// take vectors first, first + stride, ...; a bad row is reported once (by the
// thread holding its first vector) and skipped.  The new row is loaded before
// the table lookup so that its latency overlaps the lookup's two dependent
// loads (position, then table entry).
__device__ __forceinline__ void write_bf16_vectors(const WriteArgs &a, int64_t first, int64_t stride)
{
    const int32_t row_vecs = a.dims.n_kv_heads * a.dims.head_dim / 8;
    const int64_t n_vecs = (int64_t)a.n_seqs * a.n_new * row_vecs;
    const uint4 *k_new = static_cast<const uint4 *>(a.k_new);
    const uint4 *v_new = static_cast<const uint4 *>(a.v_new);
    uint4 *k_pool = static_cast<uint4 *>(a.k_pool);
    uint4 *v_pool = static_cast<uint4 *>(a.v_pool);
    const bool narrow = n_vecs <= 0x7fffffffLL;
    for (int64_t i = first; i < n_vecs; i += stride) {
        const int64_t r = index_div(i, row_vecs, narrow);
        const int32_t v = (int32_t)(i - r * row_vecs);
        const int64_t s = index_div(r, a.n_new, narrow);
        const uint4 kx = __ldcs(k_new + i);
        const uint4 vx = __ldcs(v_new + i);
        const int64_t t = (int64_t)__ldg(a.start_pos + s) + (r - s * a.n_new);
        const int64_t row = pool_row_of(a.tables + s * a.max_blocks, a.max_blocks, a.dims.n_blocks,
                                        a.dims.block_size, t, v == 0 ? a.dev_status : nullptr);
        if (row < 0) continue;
        k_pool[row * row_vecs + v] = kx;
        v_pool[row * row_vecs + v] = vx;
    }
}

// Symmetric int8 quantisation in IEEE binary32 with round-to-nearest-even
// (libmir-metal paged/mod.rs, KvPageFormat::Int8PerTokenHead): per (token,
// kv head) row of K or of V, amax by a max-reduction, scale = amax / 127
// (correctly rounded division), code = clamp(rint(x / scale), -127, 127).
//
// A warp unit is four kv heads of one token's K or V row: eight lanes per
// head, each lane holding EPL = head_dim / 8 consecutive elements.  The
// unit's new rows are loaded before the table lookup (position, then table
// entry: two dependent loads), so the three loads overlap.  Warps take units
// first, first + stride, ...; unit = (row * 2 + K/V) * head_quads + quad.
template <int EPL>
__device__ __forceinline__ void write_int8_units(const WriteArgs &a, float *k_scales, float *v_scales,
                                                 int64_t first, int64_t stride)
{
    constexpr int D = EPL * 8;
    constexpr int VECS = EPL / 8;                      // 16-byte vectors of bf16 per lane
    const int lane = threadIdx.x & 31;
    const int32_t hkv = a.dims.n_kv_heads;
    const int32_t quads = (hkv + 3) / 4;
    const int64_t n_units = (int64_t)a.n_seqs * a.n_new * 2 * quads;
    const bool narrow = n_units <= 0x7fffffffLL;
    for (int64_t u = first; u < n_units; u += stride) {
        const int64_t rw = index_div(u, quads, narrow);
        const int32_t quad = (int32_t)(u - rw * quads);
        const int which = (int)(rw & 1);
        const int64_t r = rw >> 1;                     // r = s * n_new + j
        const int32_t h = quad * 4 + (lane >> 3);
        const bool active = h < hkv;
        const int32_t part = lane & 7;                 // elements [part * EPL, (part + 1) * EPL) of the row
        float x[EPL];
        if (active) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                static_cast<const __nv_bfloat16 *>(which ? a.v_new : a.k_new) + (r * hkv + h) * D + part * EPL);
#pragma unroll
            for (int v = 0; v < VECS; ++v) {
                const uint4 raw = __ldcs(src + v);
                const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const __nv_bfloat162 p2 = *reinterpret_cast<const __nv_bfloat162 *>(&w4[k]);
                    x[8 * v + 2 * k] = __low2float(p2);
                    x[8 * v + 2 * k + 1] = __high2float(p2);
                }
            }
        } else {
#pragma unroll
            for (int e = 0; e < EPL; ++e) x[e] = 0.0f;
        }
        const int64_t s = index_div(r, a.n_new, narrow);
        const int64_t t = (int64_t)__ldg(a.start_pos + s) + (r - s * a.n_new);
        const int64_t row = pool_row_of(a.tables + s * a.max_blocks, a.max_blocks, a.dims.n_blocks,
                                        a.dims.block_size, t,
                                        lane == 0 && which == 0 && quad == 0 ? a.dev_status : nullptr);
        if (row < 0) continue;                         // the same token for the whole warp
        float amax = 0.0f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float scale = __fdiv_rn(amax, 127.0f);
        // code = rint(fl(x / scale)) without a division per element: with the
        // correctly rounded reciprocal rcp = fl(1 / scale) (scale normal), the
        // product q = fl(x * rcp) is within |x / scale| * (2^-23 + 2^-48) <= 1.53e-5
        // of x / scale (|x / scale| < 128), and fl(x / scale) within half an ulp
        // (<= 3.8e-6) of it; so when q is farther than 3e-5 from every
        // half-integer, q and fl(x / scale) round to the same integer.  The
        // rare q closer than that (a tie or a near-tie) takes the division.
        const bool fast = scale >= 1.17549435e-38f;            // normal: rcp is finite and within 2^-24
        const float rcp = fast ? __frcp_rn(scale) : 0.0f;
        int c[EPL];
        bool need_div = false;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            const float q = __fmul_rn(x[e], rcp);
            const float frac = q - floorf(q);                   // exact for |q| < 2^23
            c[e] = __float2int_rn(q);
            need_div |= !(fast && fabsf(frac - 0.5f) > 3.0e-5f);
        }
        if (__any_sync(0xffffffffu, need_div && amax != 0.0f)) {    // rare: a (near-)tie in the warp's rows
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                const float q = __fmul_rn(x[e], rcp);
                if (!(fast && fabsf(q - floorf(q) - 0.5f) > 3.0e-5f)) c[e] = __float2int_rn(__fdiv_rn(x[e], scale));
            }
        }
        if (!active) continue;
        uint32_t packed[EPL / 4];
#pragma unroll
        for (int w = 0; w < EPL / 4; ++w) {
            packed[w] = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int ce = amax != 0.0f ? max(-127, min(127, c[4 * w + k])) : 0;
                packed[w] |= (uint32_t)(ce & 0xff) << (8 * k);
            }
        }
        int8_t *dst = static_cast<int8_t *>(which ? a.v_pool : a.k_pool) + (row * hkv + h) * D + part * EPL;
        if constexpr (EPL == 16)
            *reinterpret_cast<uint4 *>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        else
            *reinterpret_cast<uint2 *>(dst) = make_uint2(packed[0], packed[1]);
        if (part == 0) (which ? v_scales : k_scales)[row * hkv + h] = scale;
    }
}

}  // namespace pkv
