// write_gather.cu -- the bandwidth kernels of the paged KV cache: native bf16
// page write, int8 quantised page write (both from write_rows.cuh), and the
// explicit gather into a contiguous [n_seqs][n_kv_heads][out_tokens][head_dim]
// view.
//
// All three are HBM-bound copies.  Token rows of the token-major pool
// ([block][slot][kv_head][head_dim]) are n_kv_heads * head_dim * 2 bytes of
// contiguous memory, so every access is a coalesced 16-byte vector.
#include "common.cuh"
#include "launch.h"
#include "write_rows.cuh"

namespace pkv {

// Launch configuration of a programmatic dependent of the previous kernel on
// the stream (its CTAs are placed while that kernel drains; the kernel waits
// for it before reading anything).
static cudaLaunchConfig_t dependent_launch(cudaLaunchAttribute (&pdl)[1], unsigned grid, unsigned threads,
                                           cudaStream_t stream)
{
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(grid);
    lc.blockDim = dim3(threads);
    lc.stream = stream;
    lc.attrs = pdl;
    lc.numAttrs = 1;
    return lc;
}

// Native bf16 write: the flat 16-byte-vector space of the new rows,
// grid-strided (write_rows.cuh).
__global__ void __launch_bounds__(256) write_bf16_kernel(const WriteArgs a)
{
    grid_dependents_launch();   // a programmatic dependent: nothing is read before the wait
    grid_dependency_wait();
    write_bf16_vectors(a, (int64_t)blockIdx.x * blockDim.x + threadIdx.x, (int64_t)gridDim.x * blockDim.x);
}

// Quantised write: four kv heads of one token's K or V row per warp unit
// (write_rows.cuh).  At most 64 registers: four resident CTAs per SM, so a
// 64 x 16-token write (512 CTAs) runs in one wave.
template <int EPL>
__global__ void __launch_bounds__(256, 4) write_int8_kernel(const WriteArgs a, float *k_scales, float *v_scales)
{
    grid_dependents_launch();   // a programmatic dependent: nothing is read before the wait
    grid_dependency_wait();
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    write_int8_units<EPL>(a, k_scales, v_scales, warp, (int64_t)gridDim.x * (blockDim.x >> 5));
}

// Gather: one warp per (sequence, kv head, logical block) unit -- block_size
// output rows of head_dim elements, contiguous in the output -- with the
// unit's indices and table entry computed once.  Each lane loads up to UNROLL
// 16-byte vectors of K and of V (zeros past the length), then stores them with
// streaming stores.  One unit per warp and no persistent loop: the CTA
// scheduler balances the equal-sized units, so no warp ends with one more
// unit than the others; 128-thread CTAs measured ~1 % faster than 256 or 512
// (16 sequences x 2048 tokens: 6012 GB/s, above a device-to-device cudaMemcpy
// of the same bytes at 5770).  Launched as a programmatic dependent, so the
// next call's CTAs take the SMs this one's last wave leaves (6430 GB/s back
// to back).
template <int UNROLL>
__global__ void __launch_bounds__(128) gather_kernel(
    const uint4 *__restrict__ k_pool, const uint4 *__restrict__ v_pool, int32_t n_blocks,
    int32_t block_size, int32_t n_kv_heads, int32_t d_shift, const int32_t *__restrict__ tables,
    int32_t max_blocks, const int32_t *__restrict__ lens, int32_t out_tokens,
    uint4 *__restrict__ k_out, uint4 *__restrict__ v_out, int32_t blocks_out, int64_t n_units, int32_t *dev_status)
{
    grid_dependents_launch();   // a programmatic dependent: nothing is read before the wait
    grid_dependency_wait();
    const int lane = threadIdx.x & 31;
    const int64_t n_warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int32_t limit = min(out_tokens, max_blocks * block_size);
    const int32_t d_vecs = 1 << d_shift;
    for (int64_t unit = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); unit < n_units;
         unit += n_warps) {
        const int32_t j = (int32_t)(unit % blocks_out);
        const int64_t sh = unit / blocks_out;                 // s * n_kv_heads + h
        const int32_t h = (int32_t)(sh % n_kv_heads);
        const int64_t s = sh / n_kv_heads;
        const int32_t len = __ldg(lens + s);
        const int32_t t0 = j * block_size;
        const int32_t rows_out = min(block_size, out_tokens - t0);
        int32_t rows_in = 0, b = 0;
        if (len < 0 || len > limit) {
            if (j == 0 && h == 0 && lane == 0) report(dev_status, PKV_DEV_BAD_LENGTH);
        } else if (len > t0) {
            rows_in = min(rows_out, len - t0);
            b = __ldg(tables + s * max_blocks + j);
            if (b < 0 || b > n_blocks) {
                if (lane == 0) report(dev_status, PKV_DEV_BAD_BLOCK_ID);
                rows_in = 0;
            }
        }
        const int64_t row_stride = (int64_t)n_kv_heads << d_shift;   // vectors between a block's token rows
        const int64_t src0 = (int64_t)b * block_size * row_stride + ((int64_t)h << d_shift);
        const int64_t dst0 = (sh * out_tokens + t0) << d_shift;
        const int32_t n_out = rows_out << d_shift, n_in = rows_in << d_shift;
        for (int32_t v0 = 0; v0 < n_out; v0 += 32 * UNROLL) {
            uint4 kv[UNROLL], vv[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int32_t v = v0 + u * 32 + lane;
                kv[u] = make_uint4(0, 0, 0, 0);
                vv[u] = kv[u];
                if (v < n_in) {
                    const int64_t src = src0 + (int64_t)(v >> d_shift) * row_stride + (v & (d_vecs - 1));
                    kv[u] = __ldg(k_pool + src);
                    vv[u] = __ldg(v_pool + src);
                }
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int32_t v = v0 + u * 32 + lane;
                if (v < n_out) {
                    __stcs(k_out + dst0 + v, kv[u]);
                    __stcs(v_out + dst0 + v, vv[u]);
                }
            }
        }
    }
}

// Block copy (the device half of copy-on-write): the index space is, per
// (source, destination) pair, the 16-byte vectors of the K block, the V block
// and, for int8 pools, the K and V scale rows of the block.
__global__ void __launch_bounds__(256) copy_blocks_kernel(uint4 *__restrict__ k_pool, uint4 *__restrict__ v_pool,
                                                          uint4 *__restrict__ k_scales, uint4 *__restrict__ v_scales,
                                                          const int2 *__restrict__ pairs, int32_t n_blocks,
                                                          int64_t block_vecs, int64_t scale_vecs, int64_t n_vecs,
                                                          int32_t *dev_status)
{
    grid_dependents_launch();   // a programmatic dependent: nothing is read before the wait
    grid_dependency_wait();
    const int64_t per_pair = 2 * block_vecs + 2 * scale_vecs;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_vecs; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t pr = i / per_pair, r = i % per_pair;
        const int2 sd = __ldg(pairs + pr);
        if (sd.x < 0 || sd.x > n_blocks || sd.y < 0 || sd.y > n_blocks) {
            if (r == 0) report(dev_status, PKV_DEV_BAD_BLOCK_ID);
            continue;
        }
        uint4 *base;
        int64_t per_block, off;
        if (r < 2 * block_vecs) {
            base = r < block_vecs ? k_pool : v_pool;
            per_block = block_vecs;
            off = r % block_vecs;
        } else {
            const int64_t q = r - 2 * block_vecs;
            base = q < scale_vecs ? k_scales : v_scales;
            per_block = scale_vecs;
            off = q % scale_vecs;
        }
        base[(int64_t)sd.y * per_block + off] = base[(int64_t)sd.x * per_block + off];
    }
}

cudaError_t launch_write_bf16(const WriteArgs &a, cudaStream_t stream)
{
    const int64_t n_vecs = (int64_t)a.n_seqs * a.n_new * (a.dims.n_kv_heads * a.dims.head_dim / 8);
    int64_t grid = (n_vecs + 255) / 256;
    if (grid > 4096) grid = 4096;
    cudaLaunchAttribute pdl[1];
    cudaLaunchConfig_t lc = dependent_launch(pdl, (unsigned)grid, 256, stream);
    return cudaLaunchKernelEx(&lc, write_bf16_kernel, a);
}

cudaError_t launch_write_int8(const WriteArgs &a, float *k_scales, float *v_scales, cudaStream_t stream)
{
    const int64_t n_units = (int64_t)a.n_seqs * a.n_new * 2 * ((a.dims.n_kv_heads + 3) / 4);
    int64_t grid = (n_units + 7) / 8;
    if (grid > 4096) grid = 4096;
    cudaLaunchAttribute pdl[1];
    cudaLaunchConfig_t lc = dependent_launch(pdl, (unsigned)grid, 256, stream);
    if (a.dims.head_dim == 128) return cudaLaunchKernelEx(&lc, write_int8_kernel<16>, a, k_scales, v_scales);
    return cudaLaunchKernelEx(&lc, write_int8_kernel<8>, a, k_scales, v_scales);
}

cudaError_t launch_gather(const GatherArgs &a, int num_sms, cudaStream_t stream)
{
    constexpr int kUnroll = 8;
    const int32_t d_shift = a.dims.head_dim == 128 ? 4 : 3;   // 16-byte vectors per row: 16 or 8
    const int32_t blocks_out = (a.out_tokens + a.dims.block_size - 1) / a.dims.block_size;
    const int64_t n_units = (int64_t)a.n_seqs * a.dims.n_kv_heads * blocks_out;
    if (n_units == 0) return cudaSuccess;
    (void)num_sms;
    int64_t grid = (n_units + 3) / 4;                         // one unit per warp, four warps per CTA
    if (grid > 0x7fffffffLL) grid = 0x7fffffffLL;
    cudaLaunchAttribute pdl[1];
    cudaLaunchConfig_t lc = dependent_launch(pdl, (unsigned)grid, 128, stream);
    return cudaLaunchKernelEx(&lc, gather_kernel<kUnroll>, (const uint4 *)a.k_pool, (const uint4 *)a.v_pool,
                              a.dims.n_blocks, a.dims.block_size, a.dims.n_kv_heads, d_shift, a.tables,
                              a.max_blocks, a.lens, a.out_tokens, (uint4 *)a.k_out, (uint4 *)a.v_out, blocks_out,
                              n_units, a.dev_status);
}

cudaError_t launch_copy_blocks(const int32_t *pairs, int32_t n_pairs, void *k_pool, void *v_pool, float *k_scales,
                               float *v_scales, bool int8, const pkv_dims &d, int32_t *dev_status, int num_sms,
                               cudaStream_t stream)
{
    const int64_t elems = (int64_t)d.block_size * d.n_kv_heads * d.head_dim;
    const int64_t block_vecs = elems * (int8 ? 1 : 2) / 16;
    const int64_t scale_vecs = int8 ? (int64_t)d.block_size * d.n_kv_heads * 4 / 16 : 0;
    const int64_t n_vecs = (int64_t)n_pairs * (2 * block_vecs + 2 * scale_vecs);
    if (n_vecs == 0) return cudaSuccess;
    int64_t grid = (n_vecs + 255) / 256, cap = (int64_t)num_sms * 8;
    if (grid > cap) grid = cap;
    cudaLaunchAttribute pdl[1];
    cudaLaunchConfig_t lc = dependent_launch(pdl, (unsigned)grid, 256, stream);
    return cudaLaunchKernelEx(&lc, copy_blocks_kernel, (uint4 *)k_pool, (uint4 *)v_pool, (uint4 *)k_scales,
                              (uint4 *)v_scales, (const int2 *)pairs, d.n_blocks, block_vecs, scale_vecs, n_vecs,
                              dev_status);
}

}  // namespace pkv
