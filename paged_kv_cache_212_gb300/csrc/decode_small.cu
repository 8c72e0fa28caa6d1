// decode_small.cu -- the decode step for batches that fit in one wave of CTAs
// with short contexts (tiny-llm paged_kv.py's decode step: write this step's
// rows at (table[t // block_size], t % block_size), then attend the first
// ctx_len tokens through the table).  The split-KV path spends three chained
// launches (plan, split, merge) on such a batch; here one launch does it all:
// one CTA per (sequence, kv head) writes that head's new rows, then computes
// the G query heads' attention over the head's whole context -- scores into
// shared memory, a two-pass softmax, then P V -- in fp32.  Every CTA reads
// only its own kv head, so the rows it wrote are the only new ones it reads
// (visible to the block after a barrier); no CTA depends on another.
#include <math.h>

#include "common.cuh"
#include "decode_small.h"

namespace pkv {
namespace {

constexpr int kThreads = 512;
constexpr int kMaxG = 8;

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w)
{
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem)
                 : "memory");
}

// Shared-memory layout for a context of at most cap tokens:
//   kbuf [cap][D * 2 + 16] bytes (padded rows: the per-token dot products read
//   the same column of consecutive rows), vbuf [cap][D * 2], sc float [kMaxG][cap],
//   qs float [kMaxG][D], part float [kThreads * 2][kMaxG] (the P V partials of
//   the token groups: GROUPS * D = kThreads * 2 for VEC = 2).
constexpr int kPartFloats = kThreads * 2 * kMaxG;

template <int D>
__host__ __device__ constexpr size_t small_smem_bytes(int cap)
{
    return (size_t)cap * (D * 2 + 16) + (size_t)cap * D * 2 + (size_t)kMaxG * cap * 4 + (size_t)kMaxG * D * 4 +
           (size_t)kPartFloats * 4;
}

template <int D>
__global__ void __launch_bounds__(kThreads) decode_small_kernel(const DecodeArgs a, const WriteArgs w, int do_write,
                                                                 int cap)
{
    constexpr int VEC = 2;                    // head-dim elements per thread in the P V pass
    constexpr int TPT = D / VEC;              // threads per token in the P V pass
    constexpr int GROUPS = kThreads / TPT;    // tokens in flight in the P V pass
    constexpr int DV = D / 8;                 // 16-byte vectors per (token, head) row
    constexpr int KROW = D * 2 + 16;          // padded K row in shared memory (bytes)
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t *kbuf = smem;
    uint8_t *vbuf = kbuf + (size_t)cap * KROW;
    float *sc = reinterpret_cast<float *>(vbuf + (size_t)cap * D * 2);   // scores, then probabilities
    float *qs = sc + kMaxG * cap;
    float *part = qs + kMaxG * D;             // [GROUPS][kMaxG][D]
    static_assert(GROUPS * kMaxG * D == kPartFloats, "P V partials fill their region");
    __shared__ int32_t tbl[kSmallMaxBlocks];
    __shared__ float red[kThreads / 32][kMaxG];
    __shared__ float row_m[kMaxG], row_l[kMaxG];

    const int hkv = a.dims.n_kv_heads, bs = a.dims.block_size;
    const int s = blockIdx.x / hkv, h = blockIdx.x % hkv;
    const int G = a.n_q_heads / hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t *trow = a.tables + (int64_t)s * a.max_blocks;

    // 1. this step's rows of this kv head (fused decode step)
    if (do_write) {
        const uint4 *kn = static_cast<const uint4 *>(w.k_new), *vn = static_cast<const uint4 *>(w.v_new);
        uint4 *kp = static_cast<uint4 *>(w.k_pool), *vp = static_cast<uint4 *>(w.v_pool);
        for (int i = tid; i < w.n_new * DV; i += kThreads) {
            const int j = i / DV, v = i % DV;
            const int64_t t = (int64_t)__ldg(w.start_pos + s) + j;
            int32_t b = -1;
            if (t < 0 || t / bs >= w.max_blocks) {
                if (v == 0 && h == 0) report(w.dev_status, PKV_DEV_BAD_POSITION);
            } else {
                b = __ldg(trow + t / bs);
                if (b < 0 || b > w.dims.n_blocks) {
                    if (v == 0 && h == 0) report(w.dev_status, PKV_DEV_BAD_BLOCK_ID);
                    b = -1;
                }
            }
            if (b < 0) continue;
            const int64_t src = (((int64_t)s * w.n_new + j) * hkv + h) * DV + v;
            const int64_t dst = (((int64_t)b * bs + t % bs) * hkv + h) * DV + v;
            kp[dst] = __ldcs(kn + src);
            vp[dst] = __ldcs(vn + src);
        }
        __threadfence_block();
        __syncthreads();   // the rows written above are visible to the whole block
    }

    // 2. context length, table row (bad ids mark their block's tokens as absent), queries
    int32_t L = __ldg(a.ctx_lens + s);
    if (L < 0 || (int64_t)L > (int64_t)a.max_blocks * bs) {
        if (tid == 0 && h == 0) report(a.dev_status, PKV_DEV_BAD_LENGTH);
        L = 0;
    }
    const int nb = (L + bs - 1) / bs;
    for (int b = tid; b < nb; b += kThreads) {
        int32_t id = __ldg(trow + b);
        if (id < 0 || id > a.dims.n_blocks) {
            report(a.dev_status, PKV_DEV_BAD_BLOCK_ID);
            id = -1;
        }
        tbl[b] = id;
    }
    const __nv_bfloat16 *q = static_cast<const __nv_bfloat16 *>(a.q) + ((int64_t)s * a.n_q_heads + (int64_t)h * G) * D;
    for (int i = tid; i < G * D; i += kThreads) qs[i] = __bfloat162float(q[i]);
    __syncthreads();

    // 3. the whole context's K and V rows of this head into shared memory, all
    //    copies in flight at once (one memory round trip)
    {
        const uint4 *kpool = static_cast<const uint4 *>(a.k_pool), *vpool = static_cast<const uint4 *>(a.v_pool);
        for (int i = tid; i < L * DV; i += kThreads) {
            const int t = i / DV, v = i % DV;
            const int32_t b = tbl[t / bs];
            if (b < 0) continue;
            const int64_t src = (((int64_t)b * bs + t % bs) * hkv + h) * DV + v;
            cp_async16(kbuf + (size_t)t * KROW + v * 16, kpool + src);
            cp_async16(vbuf + (size_t)t * D * 2 + v * 16, vpool + src);
        }
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();

    // 4. scores in log2 units: thread per token, the G dot products over D
    const float scale_log2 = a.softmax_scale * 1.4426950408889634f;
    float pm[kMaxG];
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) pm[g] = -INFINITY;
    for (int t = tid; t < L; t += kThreads) {
        const bool present = tbl[t / bs] >= 0;
        float dot[kMaxG];
#pragma unroll
        for (int g = 0; g < kMaxG; ++g) dot[g] = 0.f;
        if (present) {
            const uint4 *krow = reinterpret_cast<const uint4 *>(kbuf + (size_t)t * KROW);
#pragma unroll 4
            for (int v = 0; v < DV; ++v) {
                const uint4 x = krow[v];
                const float2 f[4] = {bf16x2_to_float2(x.x), bf16x2_to_float2(x.y), bf16x2_to_float2(x.z),
                                     bf16x2_to_float2(x.w)};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
#pragma unroll
                    for (int g = 0; g < kMaxG; ++g)
                        if (g < G)
                            dot[g] = fmaf(f[e].y, qs[g * D + 8 * v + 2 * e + 1],
                                          fmaf(f[e].x, qs[g * D + 8 * v + 2 * e], dot[g]));
                }
            }
        }
#pragma unroll
        for (int g = 0; g < kMaxG; ++g) {
            if (g < G) {
                const float x = present ? dot[g] * scale_log2 : -INFINITY;
                sc[g * cap + t] = x;
                pm[g] = fmaxf(pm[g], x);
            }
        }
    }
    // 5. row maxima, then probabilities and row sums (block reductions)
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) {
        float x = pm[g];
        for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
        if (lane == 0) red[warp][g] = x;
    }
    __syncthreads();
    if (tid < kMaxG) {
        float x = red[0][tid];
        for (int k = 1; k < kThreads / 32; ++k) x = fmaxf(x, red[k][tid]);
        row_m[tid] = x;
    }
    __syncthreads();
    float ps[kMaxG];
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) ps[g] = 0.f;
    for (int t = tid; t < L; t += kThreads) {
#pragma unroll
        for (int g = 0; g < kMaxG; ++g) {
            if (g < G) {
                const float x = sc[g * cap + t];
                const float p = x == -INFINITY ? 0.f : exp2f(x - row_m[g]);
                sc[g * cap + t] = p;
                ps[g] += p;
            }
        }
    }
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) {
        float x = ps[g];
        for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
        if (lane == 0) red[warp][g] = x;
    }
    __syncthreads();
    if (tid < kMaxG) {
        float x = 0.f;
        for (int k = 0; k < kThreads / 32; ++k) x += red[k][tid];
        row_l[tid] = x;
    }
    __syncthreads();

    // 6. O = P V from shared memory: GROUPS tokens at a time, VEC head-dim
    //    elements per thread (absent tokens are skipped: their rows were not loaded)
    const int grp = tid / TPT, d0 = (tid % TPT) * VEC;
    float acc[kMaxG][VEC];
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) acc[g][0] = acc[g][1] = 0.f;
    for (int t = grp; t < L; t += GROUPS) {
        if (tbl[t / bs] < 0) continue;
        const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(vbuf + ((size_t)t * D + d0) * 2));
#pragma unroll
        for (int g = 0; g < kMaxG; ++g) {
            if (g < G) {
                const float p = sc[g * cap + t];
                acc[g][0] = fmaf(p, v.x, acc[g][0]);
                acc[g][1] = fmaf(p, v.y, acc[g][1]);
            }
        }
    }
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) {
        if (g < G) {
            part[(grp * kMaxG + g) * D + d0] = acc[g][0];
            part[(grp * kMaxG + g) * D + d0 + 1] = acc[g][1];
        }
    }
    __syncthreads();
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out) + ((int64_t)s * a.n_q_heads + (int64_t)h * G) * D;
    for (int i = tid; i < G * D; i += kThreads) {
        const int g = i / D, d = i % D;
        float o = 0.f;
        for (int k = 0; k < GROUPS; ++k) o += part[(k * kMaxG + g) * D + d];
        const float l = row_l[g];
        out[i] = __float2bfloat16_rn(l > 0.f ? o / l : 0.f);
    }
    if (a.lse_out && tid < G) {
        const float l = row_l[tid];
        a.lse_out[(int64_t)s * a.n_q_heads + (int64_t)h * G + tid] =
            l > 0.f ? (row_m[tid] + log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
}

}  // namespace

int small_max_tokens(int head_dim) { return kSmallKVBytes / (4 * head_dim); }

bool decode_small_eligible(const DecodeArgs &a, int num_sms)
{
    const int G = a.n_q_heads / a.dims.n_kv_heads;
    return a.kv_dtype == PKV_KV_BF16 && a.split_tokens == 0 && G <= kMaxG &&
           (int64_t)a.n_seqs * a.dims.n_kv_heads <= num_sms &&
           (int64_t)a.max_blocks * a.dims.block_size <= small_max_tokens(a.dims.head_dim);
}

cudaError_t launch_decode_small(const DecodeArgs &a, const WriteArgs *write, cudaStream_t stream)
{
    const unsigned grid = (unsigned)(a.n_seqs * a.dims.n_kv_heads);
    const WriteArgs w = write ? *write : WriteArgs{};
    const int cap = a.max_blocks * a.dims.block_size;      // tokens the buffers hold
    // the shared memory limit belongs to the current device: set per device
    const size_t smem = a.dims.head_dim == 128 ? small_smem_bytes<128>(cap) : small_smem_bytes<64>(cap);
    const cudaError_t attr_err =
        a.dims.head_dim == 128
            ? prepare_kernel(reinterpret_cast<const void *>(decode_small_kernel<128>), kThreads, smem, nullptr)
            : prepare_kernel(reinterpret_cast<const void *>(decode_small_kernel<64>), kThreads, smem, nullptr);
    if (attr_err != cudaSuccess) return attr_err;
    if (a.dims.head_dim == 128)
        decode_small_kernel<128><<<grid, kThreads, smem, stream>>>(a, w, write ? 1 : 0, cap);
    else
        decode_small_kernel<64><<<grid, kThreads, smem, stream>>>(a, w, write ? 1 : 0, cap);
    return cudaGetLastError();
}

}  // namespace pkv
