// decode_small.cu -- the decode step for batches that fit in one wave of CTAs
// with short contexts (tiny-llm paged_kv.py's decode step: write this step's
// rows at (table[t // block_size], t % block_size), then attend the first
// ctx_len tokens through the table).  The split-KV path spends three chained
// launches (plan, split, merge) on such a batch; here one launch does it all:
// one CTA per (sequence, kv head) writes that head's new rows, then computes
// the G query heads' attention over the head's whole context -- K Q^T on
// mma.sync (bf16 in, fp32 accumulate) into shared memory, a two-pass softmax
// in fp32, then V^T P^T on mma.sync (P rounded to bf16, as in the split-KV
// kernel).  Every CTA reads
// only its own kv head, so the rows it wrote are the only new ones it reads
// (visible to the block after a barrier); no CTA depends on another.  The
// launch is a programmatic dependent of the previous kernel on the stream (its
// CTAs are placed while that kernel drains and read nothing before it has
// completed), and lets the next one be placed the same way.
#include <math.h>

#include "common.cuh"
#include "decode_small.h"

namespace pkv {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxG = 8;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem)
                 : "memory");
}

// Shared-memory layout for a context of at most cap tokens (a multiple of 16):
//   kbuf, vbuf [cap][D * 2 + 16] bytes: K and V rows, padded by 16 bytes so
//   that an ldmatrix of 8 consecutive rows touches every bank once;
//   sc float [kMaxG][cap]: scores, then probabilities;
//   qb [kMaxG][D * 2 + 16] bytes: the query rows (bf16, rows >= G zero);
//   part float [kWarps][16][kMaxG]: each warp's 16 x 8 block of O^T.
template <int D>
__host__ __device__ constexpr int small_row_bytes() { return D * 2 + 16; }

template <int D>
__host__ __device__ constexpr size_t small_smem_bytes(int cap)
{
    return 2 * (size_t)cap * small_row_bytes<D>() + (size_t)kMaxG * cap * 4 + (size_t)kMaxG * small_row_bytes<D>() +
           (size_t)kWarps * 16 * kMaxG * 4;
}

template <int D>
__global__ void __launch_bounds__(kThreads) decode_small_kernel(const DecodeArgs a, const WriteArgs w, int do_write,
                                                                 int cap)
{
    constexpr int DV = D / 8;                         // 16-byte vectors per (token, head) row
    constexpr int ROW = small_row_bytes<D>();
    constexpr int MT = D / 16;                        // 16-row blocks of O^T (head_dim)
    constexpr int KS = kWarps / MT;                   // warps sharing one block (token split)
    static_assert(kWarps % MT == 0, "warps split evenly over the head_dim blocks");
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t *kbuf = smem;
    uint8_t *vbuf = kbuf + (size_t)cap * ROW;
    float *sc = reinterpret_cast<float *>(vbuf + (size_t)cap * ROW);
    uint8_t *qb = reinterpret_cast<uint8_t *>(sc + kMaxG * cap);
    float *part = reinterpret_cast<float *>(qb + kMaxG * ROW);
    __shared__ int32_t tbl[kSmallMaxBlocks];
    __shared__ float red[kWarps][kMaxG];
    __shared__ float row_m[kMaxG], row_l[kMaxG];

    const int hkv = a.dims.n_kv_heads, bs = a.dims.block_size;
    const int s = blockIdx.x / hkv, h = blockIdx.x % hkv;
    const int G = a.n_q_heads / hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g4 = lane >> 2, q4 = lane & 3;          // mma fragment row group / column pair
    const int mi = lane >> 3, ri = lane & 7;          // ldmatrix matrix / row within it
    const int32_t *trow = a.tables + (int64_t)s * a.max_blocks;

    // launched as a programmatic dependent: the next kernel on the stream may
    // become resident now (it waits for this grid itself); nothing is read
    // before the preceding grid has completed
    grid_dependents_launch();
    grid_dependency_wait();

    // 1. context length, table row (bad ids mark their block's tokens as
    //    absent) and query rows; they do not depend on this step's rows
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
    {
        const uint4 *q = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(a.q) +
                                                         ((int64_t)s * a.n_q_heads + (int64_t)h * G) * D);
        for (int i = tid; i < kMaxG * DV; i += kThreads) {
            const int g = i / DV, v = i % DV;
            *reinterpret_cast<uint4 *>(qb + g * ROW + v * 16) = g < G ? __ldg(q + g * DV + v) : make_uint4(0, 0, 0, 0);
        }
    }

    // 2. this step's rows of this kv head (fused decode step)
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
    }
    __syncthreads();   // table, queries and the rows written above are visible to the whole block

    // 3. the whole context's K and V rows of this head into shared memory, all
    //    copies in flight at once (one memory round trip); V rows of absent
    //    tokens up to the next multiple of 16 are zeroed (0 x NaN must not
    //    reach O through the products)
    const int n_tiles = (L + 15) / 16;
    {
        const uint4 *kpool = static_cast<const uint4 *>(a.k_pool), *vpool = static_cast<const uint4 *>(a.v_pool);
        for (int i = tid; i < n_tiles * 16 * DV; i += kThreads) {
            const int t = i / DV, v = i % DV;
            const int32_t b = t < L ? tbl[t / bs] : -1;
            if (b < 0) {
                *reinterpret_cast<uint4 *>(vbuf + (size_t)t * ROW + v * 16) = make_uint4(0, 0, 0, 0);
                continue;
            }
            const int64_t src = (((int64_t)b * bs + t % bs) * hkv + h) * DV + v;
            cp_async16(kbuf + (size_t)t * ROW + v * 16, kpool + src);
            cp_async16(vbuf + (size_t)t * ROW + v * 16, vpool + src);
        }
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();

    // 4. scores S^T = K Q^T in log2 units, one 16-token tile per warp at a time
    //    (mma.sync m16n8k16: tokens as M, the query heads padded to 8 as N);
    //    scores of absent tokens and padding heads are -inf / not stored
    const float scale_log2 = a.softmax_scale * 1.4426950408889634f;
    float pm0 = -INFINITY, pm1 = -INFINITY;           // running maxima of heads 2 q4, 2 q4 + 1
    {
        uint32_t qf[D / 16][2];                       // Q^T B fragments of every k-step
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint8_t *qr = qb + g4 * ROW + (16 * kk + 2 * q4) * 2;
            qf[kk][0] = *reinterpret_cast<const uint32_t *>(qr);
            qf[kk][1] = *reinterpret_cast<const uint32_t *>(qr + 16);
        }
        for (int tile = warp; tile < n_tiles; tile += kWarps) {
            const int t0 = tile * 16;
            float c[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t kaddr = smem_u32(kbuf) + (uint32_t)(t0 + ri + 8 * (mi & 1)) * ROW + 16u * (mi >> 1);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t af[4];
                ldmatrix_x4(af, kaddr + 32u * kk);
                mma_bf16_16816(c, af, qf[kk][0], qf[kk][1]);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int t = t0 + g4 + 8 * (e >> 1), g = 2 * q4 + (e & 1);
                const bool present = t < L && tbl[t / bs] >= 0;
                const float x = present ? c[e] * scale_log2 : -INFINITY;
                if (g < G) sc[g * cap + t] = x;
                if (e & 1)
                    pm1 = fmaxf(pm1, x);
                else
                    pm0 = fmaxf(pm0, x);
            }
        }
    }
    // 5. row maxima, then probabilities and row sums (block reductions); the
    //    probabilities cover the whole tiles (absent tokens get 0)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        pm0 = fmaxf(pm0, __shfl_xor_sync(0xffffffffu, pm0, off));
        pm1 = fmaxf(pm1, __shfl_xor_sync(0xffffffffu, pm1, off));
    }
    if (lane < 4) {
        red[warp][2 * lane] = pm0;
        red[warp][2 * lane + 1] = pm1;
    }
    __syncthreads();
    if (tid < kMaxG) {
        float x = red[0][tid];
        for (int k = 1; k < kWarps; ++k) x = fmaxf(x, red[k][tid]);
        row_m[tid] = x;
    }
    __syncthreads();
    float ps[kMaxG];
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) ps[g] = 0.f;
    for (int t = tid; t < n_tiles * 16; t += kThreads) {
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
        for (int k = 0; k < kWarps; ++k) x += red[k][tid];
        row_l[tid] = x;
    }

    // 6. O^T = V^T P^T (mma.sync: head_dim as M, heads as N, tokens as K): warp
    //    w takes head_dim block w % MT and every KS-th tile from w / MT; the KS
    //    partial blocks are summed through shared memory
    {
        const int mt = warp % MT, ks = warp / MT;
        float o[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t vaddr = smem_u32(vbuf) + (uint32_t)(ri + 8 * (mi >> 1)) * ROW + (uint32_t)(mt * 16 + 8 * (mi & 1)) * 2;
        for (int tile = ks; tile < n_tiles; tile += KS) {
            const int t0 = tile * 16;
            uint32_t af[4];
            ldmatrix_x4_trans(af, vaddr + (uint32_t)t0 * ROW);
            uint32_t b0 = 0u, b1 = 0u;
            if (g4 < G) {
                const float *pr = sc + g4 * cap + t0 + 2 * q4;
                b0 = pack_bf16x2(pr[0], pr[1]);
                b1 = pack_bf16x2(pr[8], pr[9]);
            }
            mma_bf16_16816(o, af, b0, b1);
        }
        float *pw = part + warp * 16 * kMaxG;
        pw[g4 * kMaxG + 2 * q4] = o[0];
        pw[g4 * kMaxG + 2 * q4 + 1] = o[1];
        pw[(g4 + 8) * kMaxG + 2 * q4] = o[2];
        pw[(g4 + 8) * kMaxG + 2 * q4 + 1] = o[3];
    }
    __syncthreads();
    __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out) + ((int64_t)s * a.n_q_heads + (int64_t)h * G) * D;
    for (int i = tid; i < G * D; i += kThreads) {
        const int g = i / D, d = i % D, mt = d / 16, r = d % 16;
        float o = 0.f;
#pragma unroll
        for (int k = 0; k < KS; ++k) o += part[((k * MT + mt) * 16 + r) * kMaxG + g];
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
    // a programmatic dependent of the previous kernel on the stream: its CTAs
    // are placed while that kernel drains and wait for it in the kernel
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(grid);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    lc.attrs = pdl;
    lc.numAttrs = 1;
    const int do_write = write ? 1 : 0;
    if (a.dims.head_dim == 128) return cudaLaunchKernelEx(&lc, decode_small_kernel<128>, a, w, do_write, cap);
    return cudaLaunchKernelEx(&lc, decode_small_kernel<64>, a, w, do_write, cap);
}

}  // namespace pkv
