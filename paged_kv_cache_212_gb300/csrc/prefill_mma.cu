// prefill_mma.cu -- chunked paged prefill attention on the warp-level tensor
// cores (mma.sync), used for shapes the tcgen05 kernel does not take.
//
// CTA = (sequence, kv head, tile of 64 query rows).  The rows of a tile pack
// the G query heads of the kv head: row r is (chunk position p0 + r / G,
// query head g*G + r % G), so every K/V page streamed from the pool is used
// by all G heads.  A producer warp streams the sequence's keys 16 at a time
// (one TMA box per 64-column half of K and of V, through the block table)
// into a shared-memory ring; four consumer warps own 16 rows each and run
// S = Q K^T, an online softmax, and O += P V with m16n8k16 bf16 mma.sync.
// Query position P + p (P = prefix length) sees keys 0 .. P + p (metrale
// impl_more.rs: a query at q_pos attends only slots <= q_pos of its block).
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {

namespace {

constexpr int kRows = 64;       // query rows per CTA
constexpr int kKeys = 16;       // keys per stage
constexpr int kStagesP = 8;

struct PrefillParams {
    const __nv_bfloat16 *q;
    int32_t n_q_heads, group, chunk;
    int32_t n_blocks, block_size;
    const int32_t *tables;
    int32_t max_blocks;
    const int32_t *prefix_lens;
    float scale_log2;
    __nv_bfloat16 *out;
    float *lse_out;
    int32_t *dev_status;
    int32_t tiles_per_seq;
};

__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t chunk)
{
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(160, 1) prefill_mma_kernel(const __grid_constant__ CUtensorMap q_map,
                                                             const __grid_constant__ CUtensorMap k_map,
                                                             const __grid_constant__ CUtensorMap v_map,
                                                             const PrefillParams p)
{
    constexpr int HALVES = D / 64;
    constexpr int KSTEPS = D / 16;
    constexpr int NT = D / 8;                                   // n-tiles of the output
    constexpr uint32_t kTileHalf = kKeys * 128u;                // one 64-column half of 16 keys
    constexpr uint32_t kStageBytes = 2u * HALVES * kTileHalf;   // K and V
    constexpr uint32_t kQHalf = kRows * 128u;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *q_smem = base;
    uint8_t *stages = base + HALVES * kQHalf;
    uint64_t *full_bar = reinterpret_cast<uint64_t *>(stages + kStagesP * kStageBytes);
    uint64_t *empty_bar = full_bar + kStagesP;
    uint64_t *q_bar = empty_bar + kStagesP;
    volatile int32_t *abort_flag = reinterpret_cast<int32_t *>(q_bar + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x % p.tiles_per_seq;
    const int kvh = blockIdx.y;
    const int s = blockIdx.z;
    const int G = p.group;
    const int pos_per_tile = kRows / G;
    const int p0 = tile * pos_per_tile;
    const int p_last = min(p0 + pos_per_tile, p.chunk) - 1;
    const int32_t P = __ldg(p.prefix_lens + s);
    const int32_t n_keys = P + p_last + 1;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStagesP; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], 4);
        }
        mbar_init(q_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (P < 0 || (int64_t)n_keys > (int64_t)p.max_blocks * p.block_size) {
        if (threadIdx.x == 0) report(p.dev_status, PKV_DEV_BAD_LENGTH);
        return;
    }
    const int n_kb = (n_keys + kKeys - 1) / kKeys;

    if (warp == 4) {
        if (lane == 0) {
            mbar_arrive_expect_tx(q_bar, HALVES * kQHalf);
            for (int h = 0; h < HALVES; ++h)
                tma_load_3d(q_smem + h * kQHalf, &q_map, h * 64, kvh * G, s * p.chunk + p0, q_bar);
            const int32_t *trow = p.tables + (int64_t)s * p.max_blocks;
            for (int kb = 0; kb < n_kb; ++kb) {
                const int st = kb % kStagesP;
                if (!mbar_wait(&empty_bar[st], ((kb / kStagesP) & 1) ^ 1, abort_flag)) {
                    report(p.dev_status, PKV_DEV_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                const int t = kb * kKeys;
                const int32_t blk = __ldg(trow + t / p.block_size);
                uint8_t *stg = stages + st * kStageBytes;
                if (blk < 0 || blk > p.n_blocks) {
                    // keep the ring moving; the rows stay stale and the status says so
                    report(p.dev_status, PKV_DEV_BAD_BLOCK_ID);
                    mbar_arrive(&full_bar[st]);
                    continue;
                }
                const int32_t row0 = blk * p.block_size + t % p.block_size;
                mbar_arrive_expect_tx(&full_bar[st], kStageBytes);
                for (int h = 0; h < HALVES; ++h) {
                    tma_load_3d(stg + h * kTileHalf, &k_map, h * 64, kvh, row0, &full_bar[st]);
                    tma_load_3d(stg + (HALVES + h) * kTileHalf, &v_map, h * 64, kvh, row0, &full_bar[st]);
                }
            }
            if (*abort_flag) {
                const int first = n_kb > kStagesP ? n_kb - kStagesP : 0;
                for (int i = first; i < n_kb; ++i) (void)mbar_wait(&full_bar[i % kStagesP], (i / kStagesP) & 1);
                (void)mbar_wait(q_bar, 0);
            }
        }
        return;
    }

    // ---------------- consumer warps: 16 query rows each ----------------
    const int g = lane >> 2, qd = lane & 3;
    const int mi = lane >> 3, ri = lane & 7;
    if (!__all_sync(0xffffffffu, mbar_wait(q_bar, 0, abort_flag))) {
        if (lane == 0) report(p.dev_status, PKV_DEV_TIMEOUT);
        *abort_flag = 1;
        return;
    }
    // Q A-fragments for this warp's rows, kept in registers
    uint32_t qa[KSTEPS][4];
    {
        const uint32_t qb = smem_u32(q_smem);
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
            const uint32_t row = (uint32_t)(warp * 16 + ri + 8 * (mi & 1));
            const uint32_t chunk = (uint32_t)((kk % 4) * 2 + (mi >> 1));
            ldmatrix_x4(qa[kk], qb + (uint32_t)(kk / 4) * kQHalf + swz128(row, chunk));
        }
    }
    // absolute positions of this thread's two rows
    const int r0 = warp * 16 + g, r1 = r0 + 8;
    const int32_t qpos0 = P + p0 + r0 / G, qpos1 = P + p0 + r1 / G;
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const int32_t min_qpos = P + p0 + (warp * 16) / G;   // smallest position among the warp's rows

    for (int kb = 0; kb < n_kb; ++kb) {
        const int st = kb % kStagesP;
        if (!__all_sync(0xffffffffu, mbar_wait(&full_bar[st], (kb / kStagesP) & 1, abort_flag))) {
            if (lane == 0) report(p.dev_status, PKV_DEV_TIMEOUT);
            *abort_flag = 1;
            return;
        }
        const uint32_t kbase = smem_u32(stages + st * kStageBytes);
        const uint32_t vbase = kbase + HALVES * kTileHalf;
        const int key0 = kb * kKeys;
        // S[16 rows x 16 keys] in two n-tiles of 8 keys
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
            // matrices: (keys 0-7, chunk c), (keys 0-7, chunk c+1), (keys 8-15, c), (keys 8-15, c+1)
            const uint32_t key = (uint32_t)(ri + 8 * (mi >> 1));
            const uint32_t chunk = (uint32_t)((kk % 4) * 2 + (mi & 1));
            uint32_t b[4];
            ldmatrix_x4(b, kbase + (uint32_t)(kk / 4) * kTileHalf + swz128(key, chunk));
            mma_bf16_16816(sc[0], qa[kk], b[0], b[1]);
            mma_bf16_16816(sc[1], qa[kk], b[2], b[3]);
        }
        const bool need_mask = key0 + kKeys - 1 > min_qpos;
        float x[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = key0 + n * 8 + 2 * qd + (e & 1);
                const int32_t qp = e < 2 ? qpos0 : qpos1;
                const float v = sc[n][e] * p.scale_log2;
                x[n][e] = (!need_mask || key <= qp) ? v : -INFINITY;
            }
        }
        float bm0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
        float bm1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 1));
        bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, 2));
        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 1));
        bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, 2));
        const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
        // a row whose keys are all masked so far keeps m = -inf; use 0 as the reference
        const float ref0 = mn0 == -INFINITY ? 0.f : mn0, ref1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = fast_exp2(m0 - ref0), al1 = fast_exp2(m1 - ref1);
        float pr[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            pr[n][0] = fast_exp2(x[n][0] - ref0);
            pr[n][1] = fast_exp2(x[n][1] - ref0);
            pr[n][2] = fast_exp2(x[n][2] - ref1);
            pr[n][3] = fast_exp2(x[n][3] - ref1);
        }
        m0 = mn0;
        m1 = mn1;
        l0 = l0 * al0 + pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1];
        l1 = l1 * al1 + pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3];
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            acc[n][0] *= al0;
            acc[n][1] *= al0;
            acc[n][2] *= al1;
            acc[n][3] *= al1;
        }
        // P as the A operand (keys as k): FA2 register reuse of the S fragments
        uint32_t pa[4];
        pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
        pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
        pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
        pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);
        // V rows past the keys this tile may see can hold anything: zero them in the fragments
        const bool tail = key0 + kKeys > n_keys;
        uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
        if (tail) {
            const int ka = key0 + 2 * qd, kb2 = key0 + 8 + 2 * qd;
            vm0 = (ka < n_keys ? 0x0000ffffu : 0u) | (ka + 1 < n_keys ? 0xffff0000u : 0u);
            vm1 = (kb2 < n_keys ? 0x0000ffffu : 0u) | (kb2 + 1 < n_keys ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int c = 0; c < NT / 2; ++c) {
            // matrices: (keys 0-7, d chunk 2c'), (keys 8-15, 2c'), (keys 0-7, 2c'+1), (keys 8-15, 2c'+1)
            const uint32_t key = (uint32_t)(ri + 8 * (mi & 1));
            const uint32_t chunk = (uint32_t)((c % 4) * 2 + (mi >> 1));
            uint32_t b[4];
            ldmatrix_x4_trans(b, vbase + (uint32_t)(c / 4) * kTileHalf + swz128(key, chunk));
            b[0] &= vm0;
            b[1] &= vm1;
            b[2] &= vm0;
            b[3] &= vm1;
            mma_bf16_16816(acc[2 * c], pa, b[0], b[1]);
            mma_bf16_16816(acc[2 * c + 1], pa, b[2], b[3]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[st]);
    }
    // finalize rows
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float inv0 = 1.f / l0, inv1 = 1.f / l1;
    const int pos0 = p0 + r0 / G, pos1 = p0 + r1 / G;
    const int h0 = kvh * G + r0 % G, h1 = kvh * G + r1 % G;
    const bool ok0 = pos0 <= p_last, ok1 = pos1 <= p_last;
    __nv_bfloat16 *o0 = p.out + (((int64_t)s * p.chunk + pos0) * p.n_q_heads + h0) * D;
    __nv_bfloat16 *o1 = p.out + (((int64_t)s * p.chunk + pos1) * p.n_q_heads + h1) * D;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        const int d = n * 8 + 2 * qd;
        if (ok0) *reinterpret_cast<uint32_t *>(o0 + d) = pack_bf16x2(acc[n][0] * inv0, acc[n][1] * inv0);
        if (ok1) *reinterpret_cast<uint32_t *>(o1 + d) = pack_bf16x2(acc[n][2] * inv1, acc[n][3] * inv1);
    }
    if (p.lse_out && qd == 0) {
        if (ok0) p.lse_out[((int64_t)s * p.chunk + pos0) * p.n_q_heads + h0] = (m0 + __log2f(l0)) * 0.69314718055994531f;
        if (ok1) p.lse_out[((int64_t)s * p.chunk + pos1) * p.n_q_heads + h1] = (m1 + __log2f(l1)) * 0.69314718055994531f;
    }
}

cudaError_t launch_prefill_mma(const PrefillArgs &a, cudaStream_t stream)
{
    const pkv_dims &d = a.dims;
    const int G = a.n_q_heads / d.n_kv_heads;
    if (64 % G != 0) return cudaErrorInvalidValue;
    PrefillParams p{};
    p.q = static_cast<const __nv_bfloat16 *>(a.q);
    p.n_q_heads = a.n_q_heads;
    p.group = G;
    p.chunk = a.chunk;
    p.n_blocks = d.n_blocks;
    p.block_size = d.block_size;
    p.tables = a.tables;
    p.max_blocks = a.max_blocks;
    p.prefix_lens = a.prefix_lens;
    p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.lse_out = a.lse_out;
    p.dev_status = a.dev_status;
    const int pos_per_tile = kRows / G;
    p.tiles_per_seq = (a.chunk + pos_per_tile - 1) / pos_per_tile;

    CUtensorMap qmap, kmap, vmap;
    {
        const uint64_t dims[3] = {(uint64_t)d.head_dim, (uint64_t)a.n_q_heads, (uint64_t)a.n_seqs * a.chunk};
        const uint64_t strides[2] = {(uint64_t)d.head_dim * 2, (uint64_t)a.n_q_heads * d.head_dim * 2};
        const uint32_t box[3] = {64u, (uint32_t)G, (uint32_t)pos_per_tile};
        if (encode_tensor_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.q), dims, strides,
                              box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const uint64_t rows = (uint64_t)(d.n_blocks + 1) * d.block_size;
    const uint64_t dims[3] = {(uint64_t)d.head_dim, (uint64_t)d.n_kv_heads, rows};
    const uint64_t strides[2] = {(uint64_t)d.head_dim * 2, (uint64_t)d.n_kv_heads * d.head_dim * 2};
    const uint32_t box[3] = {64u, 1u, 16u};
    if (encode_tensor_map(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.k_pool), dims, strides,
                          box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode_tensor_map(&vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.v_pool), dims, strides,
                          box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    const int halves = d.head_dim / 64;
    const size_t smem = 1024 + (size_t)halves * kRows * 128 + (size_t)kStagesP * 2 * halves * kKeys * 128 +
                        (2 * kStagesP + 1) * 8 + 16;
    dim3 grid((unsigned)p.tiles_per_seq, (unsigned)d.n_kv_heads, (unsigned)a.n_seqs);
    cudaError_t e;
    if (d.head_dim == 128) {
        e = cudaFuncSetAttribute(prefill_mma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        prefill_mma_kernel<128><<<grid, 160, smem, stream>>>(qmap, kmap, vmap, p);
    } else {
        e = cudaFuncSetAttribute(prefill_mma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        prefill_mma_kernel<64><<<grid, 160, smem, stream>>>(qmap, kmap, vmap, p);
    }
    return cudaGetLastError();
}

}  // namespace pkv
