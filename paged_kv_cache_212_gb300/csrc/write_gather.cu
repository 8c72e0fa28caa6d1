// write_gather.cu -- the bandwidth kernels of the paged KV cache: native bf16
// page write, int8 quantised page write, and the explicit gather into a
// contiguous [n_seqs][n_kv_heads][out_tokens][head_dim] view.
//
// All three are HBM-bound copies.  Token rows of the token-major pool
// ([block][slot][kv_head][head_dim]) are n_kv_heads * head_dim * 2 bytes of
// contiguous memory, so every access is a coalesced 16-byte vector.
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
    if (t < 0 || t / block_size >= max_blocks) {
        report(dev_status, PKV_DEV_BAD_POSITION);
        return -1;
    }
    int32_t b = __ldg(table_row + t / block_size);
    if (b < 0 || b > n_blocks) {
        report(dev_status, PKV_DEV_BAD_BLOCK_ID);
        return -1;
    }
    return (int64_t)b * block_size + t % block_size;
}

// One CTA per new token row: the K and V rows (n_kv_heads * head_dim bf16
// each) are copied with 16-byte vectors.
__global__ void __launch_bounds__(128) write_bf16_kernel(
    const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new, uint4 *__restrict__ k_pool,
    uint4 *__restrict__ v_pool, int32_t n_blocks, int32_t block_size, int32_t row_vecs,
    const int32_t *__restrict__ tables, int32_t max_blocks, const int32_t *__restrict__ start_pos,
    int32_t n_new, int64_t n_rows, int32_t *dev_status)
{
    for (int64_t r = blockIdx.x; r < n_rows; r += gridDim.x) {
        int64_t s = r / n_new;
        int64_t t = (int64_t)__ldg(start_pos + s) + (r - s * n_new);
        int64_t row = pool_row_of(tables + s * max_blocks, max_blocks, n_blocks, block_size, t,
                                  threadIdx.x == 0 ? dev_status : nullptr);
        if (row < 0) continue;
        const uint4 *ks = k_new + r * row_vecs;
        const uint4 *vs = v_new + r * row_vecs;
        uint4 *kd = k_pool + row * row_vecs;
        uint4 *vd = v_pool + row * row_vecs;
        for (int32_t i = threadIdx.x; i < row_vecs; i += blockDim.x) {
            uint4 a = __ldcs(ks + i);
            uint4 b = __ldcs(vs + i);
            kd[i] = a;
            vd[i] = b;
        }
    }
}

// Symmetric int8 quantisation of one (token, kv head) row per warp, in IEEE
// binary32 with round-to-nearest-even (libmir-metal paged/mod.rs,
// KvPageFormat::Int8PerTokenHead): amax by a warp max-reduction, scale =
// amax / 127 (correctly rounded division), code = clamp(rint(x / scale)).
// EPL = head_dim / 32 elements per lane.
template <int EPL>
__global__ void __launch_bounds__(256) write_int8_kernel(
    const __nv_bfloat16 *__restrict__ k_new, const __nv_bfloat16 *__restrict__ v_new,
    int8_t *__restrict__ k_pool, int8_t *__restrict__ v_pool, float *__restrict__ k_scales,
    float *__restrict__ v_scales, int32_t n_blocks, int32_t block_size, int32_t n_kv_heads,
    const int32_t *__restrict__ tables, int32_t max_blocks, const int32_t *__restrict__ start_pos,
    int32_t n_new, int64_t n_units, int32_t *dev_status)
{
    constexpr int D = EPL * 32;
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    // unit = ((s * n_new + j) * n_kv_heads + h) * 2 + (0: K, 1: V)
    for (int64_t u = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); u < n_units;
         u += warps) {
        const int which = (int)(u & 1);
        const int64_t rh = u >> 1;                 // (s * n_new + j) * n_kv_heads + h
        const int32_t h = (int32_t)(rh % n_kv_heads);
        const int64_t r = rh / n_kv_heads;         // s * n_new + j
        const int64_t s = r / n_new;
        const int64_t t = (int64_t)__ldg(start_pos + s) + (r - s * n_new);
        const int64_t row = pool_row_of(tables + s * max_blocks, max_blocks, n_blocks, block_size,
                                        t, lane == 0 ? dev_status : nullptr);
        if (row < 0) continue;
        const __nv_bfloat16 *src = (which ? v_new : k_new) + rh * D + lane * EPL;
        float x[EPL];
        if constexpr (EPL == 4) {
            uint2 raw = __ldcs(reinterpret_cast<const uint2 *>(src));
            __nv_bfloat162 p0 = *reinterpret_cast<__nv_bfloat162 *>(&raw.x);
            __nv_bfloat162 p1 = *reinterpret_cast<__nv_bfloat162 *>(&raw.y);
            x[0] = __low2float(p0);
            x[1] = __high2float(p0);
            x[2] = __low2float(p1);
            x[3] = __high2float(p1);
        } else {
            uint32_t raw = __ldcs(reinterpret_cast<const unsigned int *>(src));
            __nv_bfloat162 p0 = *reinterpret_cast<__nv_bfloat162 *>(&raw);
            x[0] = __low2float(p0);
            x[1] = __high2float(p0);
        }
        float amax = 0.0f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float scale = __fdiv_rn(amax, 127.0f);
        uint32_t packed = 0;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            int c = 0;
            if (amax != 0.0f) {
                c = __float2int_rn(__fdiv_rn(x[e], scale));
                c = max(-127, min(127, c));
            }
            packed |= (uint32_t)(c & 0xff) << (8 * e);
        }
        int8_t *dst = (which ? v_pool : k_pool) + (row * n_kv_heads + h) * D + lane * EPL;
        if constexpr (EPL == 4)
            *reinterpret_cast<uint32_t *>(dst) = packed;
        else
            *reinterpret_cast<uint16_t *>(dst) = (uint16_t)packed;
        if (lane == 0) (which ? v_scales : k_scales)[row * n_kv_heads + h] = scale;
    }
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

cudaError_t launch_write_bf16(const WriteArgs &a, cudaStream_t stream)
{
    const int64_t n_rows = (int64_t)a.n_seqs * a.n_new;
    const int32_t row_vecs = a.dims.n_kv_heads * a.dims.head_dim / 8;
    const int64_t grid = n_rows < (1 << 20) ? n_rows : (1 << 20);
    write_bf16_kernel<<<(unsigned)grid, 128, 0, stream>>>(
        (const uint4 *)a.k_new, (const uint4 *)a.v_new, (uint4 *)a.k_pool, (uint4 *)a.v_pool,
        a.dims.n_blocks, a.dims.block_size, row_vecs, a.tables, a.max_blocks, a.start_pos, a.n_new,
        n_rows, a.dev_status);
    return cudaGetLastError();
}

cudaError_t launch_write_int8(const WriteArgs &a, float *k_scales, float *v_scales,
                              cudaStream_t stream)
{
    const int64_t n_units = (int64_t)a.n_seqs * a.n_new * a.dims.n_kv_heads * 2;
    const int warps_per_cta = 8;
    int64_t grid = (n_units + warps_per_cta - 1) / warps_per_cta;
    if (grid > (1 << 20)) grid = 1 << 20;
    if (a.dims.head_dim == 128)
        write_int8_kernel<4><<<(unsigned)grid, 256, 0, stream>>>(
            (const __nv_bfloat16 *)a.k_new, (const __nv_bfloat16 *)a.v_new, (int8_t *)a.k_pool,
            (int8_t *)a.v_pool, k_scales, v_scales, a.dims.n_blocks, a.dims.block_size,
            a.dims.n_kv_heads, a.tables, a.max_blocks, a.start_pos, a.n_new, n_units, a.dev_status);
    else
        write_int8_kernel<2><<<(unsigned)grid, 256, 0, stream>>>(
            (const __nv_bfloat16 *)a.k_new, (const __nv_bfloat16 *)a.v_new, (int8_t *)a.k_pool,
            (int8_t *)a.v_pool, k_scales, v_scales, a.dims.n_blocks, a.dims.block_size,
            a.dims.n_kv_heads, a.tables, a.max_blocks, a.start_pos, a.n_new, n_units, a.dev_status);
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

}  // namespace pkv
