// prefill_tc.cu -- chunked paged prefill attention on the 5th-generation tensor
// cores (tcgen05 + TMEM), for head_dim 64 / 128 and GQA groups of 1..16.
//
// CTA = (sequence, kv head, tile of 128 query rows).  The rows of a tile pack
// the G query heads of the kv head: row r is (chunk position p0 + r / G, query
// head kvh * G + r % G), so each K/V tile serves all G heads.  Warp roles:
//   warps 0-3  softmax: thread r owns query row r = TMEM lane r;
//   warp 4     TMA producer: Q once, then K and V tiles of 128 keys, one
//              {64 columns, 16 keys} box per 16-key group, addressed through
//              the block table (groups past the last key read zeros);
//   warp 5     TMEM allocator and MMA issuer (one elected lane).
// Per key tile j:  S_j = Q K_j^T  (tcgen05.mma, M 128 x N 128, S in TMEM,
// double-buffered), softmax in registers (log2 units, a stale row maximum is
// kept unless it grows by more than 2^8, then the O row is rescaled in TMEM),
// P_j (bf16) to shared memory, O += P_j V_j (tcgen05.mma, V read MN-major).
// Query position P + p (P = prefix length) sees keys 0 .. P + p (metrale
// impl_more.rs: a query at q_pos attends only slots <= q_pos of its block).
#include <math.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {

namespace {

constexpr int kTM = 128;          // query rows per CTA (TMEM lanes)
constexpr int kTN = 128;          // keys per tile
constexpr int kKvStages = 2;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct PrefillTcParams {
    int32_t n_q_heads, group, chunk;
    int32_t n_blocks, block_size;
    int32_t pool_rows;            // (n_blocks + 1) * block_size: an out-of-range TMA row
    const int32_t *tables;
    int32_t max_blocks;
    const int32_t *prefix_lens;
    float scale_log2;
    __nv_bfloat16 *out;
    float *lse_out;
    int32_t *dev_status;
    int32_t tiles_per_seq;
    int32_t n_kv_heads;
};

// ---- tcgen05 helpers -------------------------------------------------------

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets, version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;          // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;          // SWIZZLE_128B
    return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, M x N, majors.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int M, int N, bool a_mn_major, bool b_mn_major)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Issue a load of 32 consecutive fp32 columns without waiting for it.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t *r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t chunk)
{
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(192, 1) prefill_tc_kernel(const __grid_constant__ CUtensorMap q_map,
                                                            const __grid_constant__ CUtensorMap k_map,
                                                            const __grid_constant__ CUtensorMap v_map,
                                                            const PrefillTcParams p)
{
    constexpr int PANELS = D / 64;                    // 64-column (128-byte) panels of a bf16 row
    constexpr uint32_t kQBytes = kTM * D * 2;         // 32 KiB at D 128
    constexpr uint32_t kKBytes = kTN * D * 2;
    constexpr uint32_t kPanelRows128 = 128u * 128u;   // one panel of 128 rows
    constexpr uint32_t kStageBytes = 2 * kKBytes;     // K then V
    constexpr uint32_t kPBytes = kTM * kTN * 2;       // P: 128 rows x 128 keys, 2 panels
    constexpr uint32_t kTmemCols = 512;
    constexpr uint32_t kOCol = 256;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *q_s = base;
    uint8_t *kv_s = q_s + kQBytes;
    uint8_t *p_s = kv_s + kKvStages * kStageBytes;   // after V: any descriptor overrun stays inside the CTA
    uint64_t *bars = reinterpret_cast<uint64_t *>(p_s + kPBytes);
    uint64_t *q_full = bars + 0;
    uint64_t *kv_full = bars + 1;                    // [2]
    uint64_t *kv_empty = bars + 3;                   // [2]
    uint64_t *s_full = bars + 5;                     // [2]
    uint64_t *s_free = bars + 7;                     // [2]
    uint64_t *p_full = bars + 9;
    uint64_t *o_done = bars + 10;
    uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(bars + 11);
    volatile int32_t *abort_flag = reinterpret_cast<int32_t *>(bars + 12);
    uint64_t *fin_bar = bars + 13;                  // all MMAs of this CTA retired

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles = p.tiles_per_seq;
    const int tile = tiles - 1 - (int)(blockIdx.x % tiles);   // heavy (late) tiles first
    const int kvh = blockIdx.y;
    const int s = blockIdx.z;
    const int G = p.group;
    const int pos_per_tile = kTM / G;
    const int p0 = tile * pos_per_tile;
    const int p_last = min(p0 + pos_per_tile, p.chunk) - 1;
    const int32_t P = __ldg(p.prefix_lens + s);
    const int32_t n_keys = P + p_last + 1;
    const bool bad_len = P < 0 || (int64_t)n_keys > (int64_t)p.max_blocks * p.block_size;
    const int n_kt = bad_len ? 0 : (n_keys + kTN - 1) / kTN;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < kKvStages; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], 4);
        }
        mbar_init(p_full, 4);
        mbar_init(o_done, 1);
        mbar_init(fin_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5) {
        // allocate TMEM: S double buffer (2 x 128 columns) + O (D columns), rounded to 512
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_base_s)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_s;
    if (bad_len && threadIdx.x == 0) report(p.dev_status, PKV_DEV_BAD_LENGTH);

    if (warp == 4 && n_kt > 0) {
        // ===================== TMA producer =====================
        if (lane == 0) {
            prefetch_tensormap(&q_map);
            prefetch_tensormap(&k_map);
            prefetch_tensormap(&v_map);
            mbar_arrive_expect_tx(q_full, kQBytes);
            for (int h = 0; h < PANELS; ++h)
                tma_load_3d(q_s + h * kPanelRows128, &q_map, h * 64, kvh * G, s * p.chunk + p0, q_full);
        }
        const int32_t *trow = p.tables + (int64_t)s * p.max_blocks;
        int issued = 0;
        for (int j = 0; j < n_kt; ++j) {
            const int st = j % kKvStages, use = j / kKvStages;
            if (lane == 0 && !mbar_wait(&kv_empty[st], (use & 1) ^ 1, abort_flag)) {
                report(p.dev_status, PKV_DEV_TIMEOUT);
                *abort_flag = 1;
            }
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
            // lanes 0..7: the pool row of each 16-key group of this tile
            int32_t row = p.pool_rows;  // out of range: the box reads zeros
            if (lane < kTN / 16) {
                const int32_t key0 = j * kTN + lane * 16;
                if (key0 < n_keys) {
                    const int32_t blk = __ldg(trow + key0 / p.block_size);
                    if (blk < 0 || blk > p.n_blocks)
                        report(p.dev_status, PKV_DEV_BAD_BLOCK_ID);
                    else
                        row = blk * p.block_size + key0 % p.block_size;
                }
            }
            uint8_t *ks = kv_s + st * kStageBytes;
            uint8_t *vs = ks + kKBytes;
            if (lane == 0) mbar_arrive_expect_tx(&kv_full[st], kStageBytes);
            for (int gq = 0; gq < kTN / 16; ++gq) {
                const int32_t rr = __shfl_sync(0xffffffffu, row, gq);
                if (lane == 0) {
                    for (int h = 0; h < PANELS; ++h) {
                        const uint32_t off = h * kPanelRows128 + gq * 16 * 128;
                        tma_load_3d(ks + off, &k_map, h * 64, kvh, rr, &kv_full[st]);
                        tma_load_3d(vs + off, &v_map, h * 64, kvh, rr, &kv_full[st]);
                    }
                }
            }
            ++issued;
        }
        // every copy this warp issued has landed before the CTA can exit
        if (lane == 0) {
            (void)mbar_wait(q_full, 0);
            for (int i = issued > kKvStages ? issued - kKvStages : 0; i < issued; ++i)
                (void)mbar_wait(&kv_full[i % kKvStages], (i / kKvStages) & 1);
        }
    } else if (warp == 5 && n_kt > 0) {
        // ===================== MMA issuer =====================
        // One lane issues S_j = Q K_j^T as soon as K_j has landed and S buffer
        // j & 1 is free, and O += P_j V_j as soon as P_j is written, whichever
        // is ready first (non-blocking polls, bounded by the wait limit).
        const uint32_t idesc_s = umma_idesc_bf16(kTM, kTN, false, false);
        const uint32_t idesc_o = umma_idesc_bf16(kTM, D, false, true);
        bool ok = true;
        if (lane == 0) {
            ok = mbar_wait(q_full, 0, abort_flag);
            const uint32_t q_addr = smem_u32(q_s), p_addr = smem_u32(p_s);
            int js = 0, jp = 0;
            unsigned long long t_last = global_timer_ns();
            uint32_t spin = 0;
            while (ok && jp < n_kt) {
                bool progressed = false;
                if (js < n_kt && js < jp + 2) {
                    const int st = js % kKvStages, b = js & 1;
                    if (mbar_test_wait(&kv_full[st], (js / kKvStages) & 1) &&
                        mbar_test_wait(&s_free[b], ((js >> 1) & 1) ^ 1)) {
                        tc_fence_after();
                        const uint32_t k_addr = smem_u32(kv_s + st * kStageBytes);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t off = (kk / 4) * kPanelRows128 + (kk % 4) * 32;
                            umma_bf16(tmem + b * kTN, umma_desc_sw128(q_addr + off, 16, 1024),
                                      umma_desc_sw128(k_addr + off, 16, 1024), idesc_s, kk > 0);
                        }
                        umma_commit(&s_full[b]);
                        ++js;
                        progressed = true;
                    }
                }
                if (jp < js && mbar_test_wait(p_full, jp & 1)) {
                    tc_fence_after();
                    const int st = jp % kKvStages;
                    const uint32_t v_addr = smem_u32(kv_s + st * kStageBytes + kKBytes);
#pragma unroll
                    for (int kk = 0; kk < kTN / 16; ++kk) {
                        // A = P (K-major, keys kk*16..), B = V (MN-major: 8-key groups 1024 B
                        // apart, 64-column panels kPanelRows128 apart)
                        const uint32_t a_off = (kk / 4) * kPanelRows128 + (kk % 4) * 32;
                        umma_bf16(tmem + kOCol, umma_desc_sw128(p_addr + a_off, 16, 1024),
                                  umma_desc_sw128(v_addr + kk * 2048, kPanelRows128, 1024), idesc_o,
                                  (jp > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(o_done);
                    umma_commit(&kv_empty[st]);
                    ++jp;
                    progressed = true;
                }
                if (progressed) {
                    spin = 0;
                    t_last = global_timer_ns();
                } else if ((++spin & 255u) == 0) {
                    if (*abort_flag || global_timer_ns() - t_last > kWaitTimeoutNs) ok = false;
                }
            }
            if (!ok) {
                report(p.dev_status, PKV_DEV_TIMEOUT);
                *abort_flag = 1;
            }
            // every MMA issued has retired before the TMEM is released
            umma_commit(fin_bar);
            (void)mbar_wait(fin_bar, 0);
        }
        __syncwarp();
    } else if (warp < 4) {
        // ===================== softmax warpgroup: row r = TMEM lane r =====================
        const int r = threadIdx.x;
        const int32_t qpos = P + p0 + r / G;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        float m = -INFINITY, l = 0.f;
        bool ok = n_kt > 0;
        for (int j = 0; j < n_kt && ok; ++j) {
            const int b = j & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(&s_full[b], (j >> 1) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            const int32_t key_base = j * kTN;
            const bool masked = key_base + kTN - 1 > qpos;
            // one pass: the whole S row into registers (four loads, one wait)
            uint32_t sv[kTN];
#pragma unroll
            for (int c = 0; c < kTN / 32; ++c) tmem_ld32_async(lane_base + b * kTN + c * 32, sv + c * 32);
            tmem_wait_ld();
            // S buffer b is read: the MMA warp may overwrite it with S_{j+2}
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[b]);
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < kTN; ++i) {
                const bool valid = !masked || key_base + i <= qpos;
                mx = fmaxf(mx, valid ? __uint_as_float(sv[i]) : -INFINITY);
            }
            mx *= p.scale_log2;
            // the previous P V product must be done: P is overwritten, O may be rescaled
            if (j > 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
            }
            float alpha = 1.f;
            if (m == -INFINITY) {
                m = mx;
            } else if (mx > m + kRescaleThreshold) {
                alpha = fast_exp2(m - mx);
                m = mx;
            }
            l *= alpha;
            // probabilities, row sum, P (bf16) to shared memory
#pragma unroll
            for (int c = 0; c < kTN / 32; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const int kidx = c * 32 + i;
                    const bool v0 = !masked || key_base + kidx <= qpos;
                    const bool v1 = !masked || key_base + kidx + 1 <= qpos;
                    const float e0 = v0 ? fast_exp2(__uint_as_float(sv[kidx]) * p.scale_log2 - m) : 0.f;
                    const float e1 = v1 ? fast_exp2(__uint_as_float(sv[kidx + 1]) * p.scale_log2 - m) : 0.f;
                    l += e0 + e1;
                    pk[i / 2] = pack_bf16x2(e0, e1);
                }
                // keys c*32 .. c*32+31 of row r: panel c/2, 16-byte chunks (c%2)*4 .. +3
                uint8_t *prow = p_s + (c / 2) * kPanelRows128;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    *reinterpret_cast<uint4 *>(prow + swz128(r, (c % 2) * 4 + q4)) =
                        make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
            }
            // O row rescale (rare: the row maximum grew by more than 2^8), after the
            // S row is dead; the next P V product is issued only after p_full below
            if (__any_sync(0xffffffffu, alpha != 1.f) && j > 0) {
                float v[32];
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    tmem_ld32(lane_base + kOCol + c * 32, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= alpha;
                    tmem_st32(lane_base + kOCol + c * 32, v);
                }
            }
            // last tile: V rows of keys past the last one may hold anything; zero them
            if (j == n_kt - 1 && (n_keys & 15) != 0) {
                const int first = n_keys - key_base, stop = ((n_keys + 15) & ~15) - key_base;
                uint8_t *vs = kv_s + (j % kKvStages) * kStageBytes + kKBytes;
                for (int i = r; i < (stop - first) * PANELS * 8; i += kTM) {
                    const int row = first + i / (PANELS * 8), pc = i % (PANELS * 8);
                    *reinterpret_cast<uint4 *>(vs + (pc / 8) * kPanelRows128 + swz128(row, pc % 8)) =
                        make_uint4(0, 0, 0, 0);
                }
            }
            fence_proxy_async_smem();   // P (and zeroed V rows) visible to the tensor core
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        if (ok && n_kt > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(o_done, (n_kt - 1) & 1, abort_flag));
            tc_fence_after();
        }
        if (ok && n_kt > 0) {
            const int pos = p0 + r / G, h = kvh * G + r % G;
            const bool store = pos <= p_last;
            const float inv = 1.f / l;
            __nv_bfloat16 *o = p.out + (((int64_t)s * p.chunk + pos) * p.n_q_heads + h) * D;
            uint32_t ov[D];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) tmem_ld32_async(lane_base + kOCol + c * 32, ov + c * 32);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(ov[c * 32 + i]);
                if (store) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint4 w;
                        w.x = pack_bf16x2(v[8 * q4 + 0] * inv, v[8 * q4 + 1] * inv);
                        w.y = pack_bf16x2(v[8 * q4 + 2] * inv, v[8 * q4 + 3] * inv);
                        w.z = pack_bf16x2(v[8 * q4 + 4] * inv, v[8 * q4 + 5] * inv);
                        w.w = pack_bf16x2(v[8 * q4 + 6] * inv, v[8 * q4 + 7] * inv);
                        *reinterpret_cast<uint4 *>(o + c * 32 + 8 * q4) = w;
                    }
                }
            }
            if (store && p.lse_out)
                p.lse_out[((int64_t)s * p.chunk + pos) * p.n_q_heads + h] = (m + __log2f(l)) * 0.69314718055994531f;
        } else if (!ok) {
            if (lane == 0) report(p.dev_status, PKV_DEV_TIMEOUT);
            *abort_flag = 1;
        }
    }
    // everyone meets here before the TMEM is released
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

}  // namespace pkv

namespace pkv {

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t stream)
{
    const pkv_dims &d = a.dims;
    const int G = a.n_q_heads / d.n_kv_heads;
    if (G > 16 || 128 % G != 0) return cudaErrorInvalidValue;
    PrefillTcParams p{};
    p.n_q_heads = a.n_q_heads;
    p.group = G;
    p.chunk = a.chunk;
    p.n_blocks = d.n_blocks;
    p.block_size = d.block_size;
    p.pool_rows = (d.n_blocks + 1) * d.block_size;
    p.tables = a.tables;
    p.max_blocks = a.max_blocks;
    p.prefix_lens = a.prefix_lens;
    p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
    p.out = static_cast<__nv_bfloat16 *>(a.out);
    p.lse_out = a.lse_out;
    p.dev_status = a.dev_status;
    p.n_kv_heads = d.n_kv_heads;
    const int pos_per_tile = kTM / G;
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

    const size_t smem = 1024 + (size_t)kTM * d.head_dim * 2 + (size_t)kKvStages * 2 * kTN * d.head_dim * 2 +
                        (size_t)kTM * kTN * 2 + 16 * sizeof(uint64_t);
    dim3 grid((unsigned)p.tiles_per_seq, (unsigned)d.n_kv_heads, (unsigned)a.n_seqs);
    cudaError_t e;
    if (d.head_dim == 128) {
        e = cudaFuncSetAttribute(prefill_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        prefill_tc_kernel<128><<<grid, 192, smem, stream>>>(qmap, kmap, vmap, p);
    } else {
        e = cudaFuncSetAttribute(prefill_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        prefill_tc_kernel<64><<<grid, 192, smem, stream>>>(qmap, kmap, vmap, p);
    }
    return cudaGetLastError();
}

}  // namespace pkv
