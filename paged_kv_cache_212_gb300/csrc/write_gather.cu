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

// Native bf16 write: the flat 16-byte-vector space of the new rows,
// grid-strided (write_rows.cuh).
__global__ void __launch_bounds__(256) write_bf16_kernel(const WriteArgs a)
{
    write_bf16_vectors(a, (int64_t)blockIdx.x * blockDim.x + threadIdx.x, (int64_t)gridDim.x * blockDim.x);
}

// Quantised write: one (token, kv head, K or V) row per warp (write_rows.cuh).
template <int EPL>
__global__ void __launch_bounds__(256) write_int8_kernel(const WriteArgs a, float *k_scales, float *v_scales)
{
    const int64_t warp = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    write_int8_units<EPL>(a, k_scales, v_scales, warp, (int64_t)gridDim.x * (blockDim.x >> 5));
}

// Gather: every thread owns up to UNROLL 16-byte output vectors, loads them all
// (from the pool, or zeros past the sequence length), then stores them.  The
// output index space is [n_seqs][n_kv_heads][out_tokens][head_dim / 8], so the
// stores are fully contiguous and each token's loads read whole 16-byte
// pieces of its pool row.
template <int UNROLL>
__global__ void __launch_bounds__(256) gather_kernel(
    const uint4 *__restrict__ k_pool, const uint4 *__restrict__ v_pool, int32_t n_blocks,
    int32_t block_size, int32_t n_kv_heads, int32_t d_vecs, const int32_t *__restrict__ tables,
    int32_t max_blocks, const int32_t *__restrict__ lens, int32_t out_tokens,
    uint4 *__restrict__ k_out, uint4 *__restrict__ v_out, int64_t n_vecs, int32_t *dev_status)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int32_t limit = min(out_tokens, max_blocks * block_size);
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; base < n_vecs;
         base += stride * UNROLL) {
        uint4 kv[UNROLL], vv[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t i = base + u * stride;
            kv[u] = make_uint4(0, 0, 0, 0);
            vv[u] = kv[u];
            if (i >= n_vecs) continue;
            const int32_t dv = (int32_t)(i % d_vecs);
            const int64_t rest = i / d_vecs;
            const int32_t t = (int32_t)(rest % out_tokens);
            const int64_t sh = rest / out_tokens;         // s * n_kv_heads + h
            const int32_t h = (int32_t)(sh % n_kv_heads);
            const int64_t s = sh / n_kv_heads;
            const int32_t len = __ldg(lens + s);
            if (len < 0 || len > limit) {
                if (t == 0 && h == 0 && dv == 0) report(dev_status, PKV_DEV_BAD_LENGTH);
                continue;
            }
            if (t >= len) continue;
            const int32_t b = __ldg(tables + s * max_blocks + t / block_size);
            if (b < 0 || b > n_blocks) {
                report(dev_status, PKV_DEV_BAD_BLOCK_ID);
                continue;
            }
            const int64_t src = (((int64_t)b * block_size + t % block_size) * n_kv_heads + h) * d_vecs + dv;
            kv[u] = __ldg(k_pool + src);
            vv[u] = __ldg(v_pool + src);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int64_t i = base + u * stride;
            if (i < n_vecs) {
                __stcs(k_out + i, kv[u]);
                __stcs(v_out + i, vv[u]);
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
    write_bf16_kernel<<<(unsigned)grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_write_int8(const WriteArgs &a, float *k_scales, float *v_scales, cudaStream_t stream)
{
    const int64_t n_units = (int64_t)a.n_seqs * a.n_new * a.dims.n_kv_heads * 2;
    int64_t grid = (n_units + 7) / 8;
    if (grid > 4096) grid = 4096;
    if (a.dims.head_dim == 128)
        write_int8_kernel<4><<<(unsigned)grid, 256, 0, stream>>>(a, k_scales, v_scales);
    else
        write_int8_kernel<2><<<(unsigned)grid, 256, 0, stream>>>(a, k_scales, v_scales);
    return cudaGetLastError();
}

cudaError_t launch_gather(const GatherArgs &a, int num_sms, cudaStream_t stream)
{
    constexpr int kUnroll = 4;
    const int32_t d_vecs = a.dims.head_dim / 8;
    const int64_t n_vecs = (int64_t)a.n_seqs * a.dims.n_kv_heads * a.out_tokens * d_vecs;
    if (n_vecs == 0) return cudaSuccess;
    int64_t want = (n_vecs + 256LL * kUnroll - 1) / (256LL * kUnroll);
    int64_t cap = (int64_t)num_sms * 8;  // 8 resident 256-thread CTAs per SM
    int64_t grid = want < cap ? want : cap;
    gather_kernel<kUnroll><<<(unsigned)grid, 256, 0, stream>>>(
        (const uint4 *)a.k_pool, (const uint4 *)a.v_pool, a.dims.n_blocks, a.dims.block_size,
        a.dims.n_kv_heads, d_vecs, a.tables, a.max_blocks, a.lens, a.out_tokens, (uint4 *)a.k_out,
        (uint4 *)a.v_out, n_vecs, a.dev_status);
    return cudaGetLastError();
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
    copy_blocks_kernel<<<(unsigned)grid, 256, 0, stream>>>((uint4 *)k_pool, (uint4 *)v_pool, (uint4 *)k_scales,
                                                           (uint4 *)v_scales, (const int2 *)pairs, d.n_blocks,
                                                           block_vecs, scale_vecs, n_vecs, dev_status);
    return cudaGetLastError();
}

}  // namespace pkv
