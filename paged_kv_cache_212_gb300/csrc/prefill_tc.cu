// prefill_tc.cu -- chunked paged prefill attention on the 5th-generation tensor
// cores (tcgen05 + TMEM), for head_dim 64 / 128 and GQA groups of 1..16.
//
// CTA = (sequence, kv head, two adjacent tiles of 128 query rows).  The rows of
// a tile pack the G query heads of the kv head: row r is (chunk position
// p0 + r / G, query head kvh * G + r % G), so every K/V tile serves 2 x 128
// rows.  Warp roles (384 threads):
//   warps 0-3, 4-7  softmax warpgroups of query tile 0 and 1: thread r of a
//                   warpgroup owns row r of its tile (= TMEM lane r);
//   warps 8, 10     TMA producers of K: both Q tiles once (warp 8), then for
//                   every tile of 128 keys half of its 16-key groups each, one
//                   {64 columns, 1 head, 16 keys} box per group and panel;
//   warp 11         TMA producer of V: one {64 columns, 16 keys, all panels}
//                   box per group (a panel-dimension view of the pool);
//   warp 9          TMEM allocator and MMA issuer (one lane).
// Groups are addressed through the block table, looked up one tile ahead;
// groups past the last key read the zero fill of an out-of-range row.  A TMA
// issue holds its warp for about a hundred cycles whatever the box size (the
// lanes of one warp issue one after the other), so the boxes of a tile are
// spread over three warps and V, whose layout allows it, takes 4 KiB boxes.
// TMEM (512 columns): per query tile, S (128 fp32 columns; P overwrites its
// first 64 columns as packed bf16 pairs) and O (head_dim columns).  For key
// tile j and query tile i:
//   S_ij = Q_i K_j^T (tcgen05.mma M 128, N 128, both operands in shared
//   memory); softmax in registers (log2 units; a stale row maximum is kept
//   unless it grows by more than 2^8, then the O row is rescaled in TMEM);
//   P_ij (bf16) back into TMEM; O_i += P_ij V_j (tcgen05.mma with A = P read
//   from TMEM, B = V MN-major in shared memory).
// At the end each softmax warpgroup writes its normalised O tile into shared
// memory (the K ring, free once the last S products have retired) and one
// thread stores it with a TMA copy per 64-column panel: one bulk operation
// instead of each thread storing its scattered 256-byte row.
// Issue order PV_0j, S_0,j+1, PV_1j, S_1,j+1: while one warpgroup computes the
// softmax of its tile the tensor core runs the other tile's two products, and
// the commit of S_i,j+1 also covers PV_ij, so O may be rescaled as soon as S is
// ready.  Keeping P in TMEM spares the shared-memory port the P round trip
// (the S and P V operand reads and the TMA writes already come close to its
// bandwidth).  Query position P + p (P = prefix length) sees keys 0 .. P + p
// (metrale impl_more.rs: a query at q_pos attends only slots <= q_pos of its
// block).
#include <math.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kTM = 128;           // query rows per tile (TMEM lanes)
constexpr int kNQ = 2;             // query tiles per CTA
constexpr int kTN = 128;           // keys per K/V tile
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTileCols = 256;        // TMEM columns per query tile: S / P, O
constexpr uint32_t kOCol = 128;            // O's column within a query tile's range

// Ring slots (one 128-key tile each) of K and of V that fit beside the Q tiles.
template <int D>
__host__ __device__ constexpr int k_slots() { return D == 128 ? 3 : 6; }
template <int D>
__host__ __device__ constexpr int v_slots() { return D == 128 ? 2 : 4; }

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
    int32_t tiles_per_seq;        // 128-row query tiles per (sequence, kv head)
    int32_t pairs_per_seq;        // CTAs per (sequence, kv head)
    int32_t n_seqs, n_kv_heads;
    unsigned long long wait_ns;   // limit of the pipeline waits
};

// Batches of at most this many sequences are scheduled longest prefix first.
constexpr int kSortMaxSeqs = 32;

// Register split (setmaxnreg): the block is launched with kLaunchRegs per
// thread; warpgroup 2 (TMA producers, MMA issuer) keeps kRegsIssue and hands
// the rest to the two softmax warpgroups, whose rows of 128 scores stay in
// registers.  The sum must not exceed what the block was launched with, or the
// increase would wait for registers that never come free.
constexpr int kLaunchRegs = 168;             // 65536 / 384, rounded down to a multiple of 8
constexpr int kRegsIssue = 72;
constexpr int kRegsSoftmax = 216;
static_assert(128 * kRegsIssue + 256 * kRegsSoftmax <= 384 * kLaunchRegs, "register split above the launch");

// ---- tcgen05 helpers -------------------------------------------------------

// The 8 products of one 128-row tile step in one asm block, so that the
// predicates are set once (first product: accumulate_first; the rest
// accumulate) rather than once per instruction.  A and B shared-memory
// descriptors (SS form).
__device__ __forceinline__ void umma_bf16_x8(uint32_t d_tmem, const uint64_t (&a)[8], const uint64_t (&b)[8],
                                             uint32_t idesc, uint32_t accumulate_first)
{
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %17, 0;\n\t"
        "setp.eq.b32 q, %17, %17;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %9, %18, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %10, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %11, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %12, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %13, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %14, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %15, %18, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %16, %18, q;\n\t}" ::"r"(d_tmem),
        "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(a[4]), "l"(a[5]), "l"(a[6]), "l"(a[7]), "l"(b[0]),
        "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]), "r"(accumulate_first),
        "r"(idesc)
        : "memory");
}

// The 8 products of one tile step in the TS form: D (TMEM) += A (TMEM, M x 16,
// K-major: lane = row, column c = bf16 pair 2c, 2c + 1; product k at a_tmem +
// 8 k) * B (shared-memory descriptor), predicates set once as above.
__device__ __forceinline__ void umma_bf16_ts_x8(uint32_t d_tmem, uint32_t a_tmem, const uint64_t (&b)[8],
                                                uint32_t idesc, uint32_t accumulate_first)
{
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t.reg .b32 a1, a2, a3, a4, a5, a6, a7;\n\t"
        "setp.ne.b32 p, %10, 0;\n\t"
        "setp.eq.b32 q, %10, %10;\n\t"
        "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\tadd.u32 a4, %1, 32;\n\t"
        "add.u32 a5, %1, 40;\n\tadd.u32 a6, %1, 48;\n\tadd.u32 a7, %1, 56;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %11, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], %3, %11, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], %4, %11, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], %5, %11, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], %6, %11, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], %7, %11, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], %8, %11, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], %9, %11, q;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]),
        "r"(accumulate_first), "r"(idesc)
        : "memory");
}

// max(a, b, c) in one instruction (sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t chunk)
{
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// Shared memory -> global through a 4-D tensor map (elements past the map's
// extent are not written), then the commit of the bulk group.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, const void *src, int32_t c0, int32_t c1,
                                             int32_t c2, int32_t c3)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];\n\t"
        "cp.async.bulk.commit_group;" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// The bulk copies this thread committed have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// AND of v over the 128 threads of a warpgroup (named barrier id); every
// thread of the warpgroup must reach it.
__device__ __forceinline__ bool wg_and(uint32_t id, bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id)
        : "memory");
    return r != 0;
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(384, 1) prefill_tc_kernel(const __grid_constant__ CUtensorMap q_map,
                                                            const __grid_constant__ CUtensorMap k_map,
                                                            const __grid_constant__ CUtensorMap v_map,
                                                            const __grid_constant__ CUtensorMap o_map,
                                                            const PrefillTcParams p)
{
    constexpr int PANELS = D / 64;                          // 64-column (128-byte) panels of a bf16 row
    constexpr int NK = k_slots<D>(), NV = v_slots<D>();
    constexpr uint32_t kQPanel = kTM * 128u;                // 16 KiB: one panel of a 128-row Q tile
    constexpr uint32_t kQTile = PANELS * kQPanel;
    constexpr uint32_t kKVPanel = kTN * 128u;               // 16 KiB: one panel of a 128-key K tile
    constexpr uint32_t kSlotBytes = PANELS * kKVPanel;      // one K or V tile
    constexpr uint32_t kVGroup = PANELS * 2048u;            // one 16-key group of a V tile (all panels)

    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *q_s = base;                                    // kNQ Q tiles
    // K tile: [panel][128 keys][128 B]; V tile: [16-key group][panel][16 keys][128 B]
    uint8_t *k_ring = q_s + kNQ * kQTile;                   // NK K tiles
    uint8_t *v_ring = k_ring + NK * kSlotBytes;             // NV V tiles
    uint64_t *bars = reinterpret_cast<uint64_t *>(v_ring + NV * kSlotBytes);
    uint64_t *q_full = bars + 0;
    uint64_t *k_full = bars + 1;                            // [NK]
    uint64_t *k_empty = k_full + NK;                        // [NK]
    uint64_t *v_full = k_empty + NK;                        // [NV]
    uint64_t *v_empty = v_full + NV;                        // [NV]
    uint64_t *s_full = v_empty + NV;                        // [kNQ]: S_ij in TMEM (and PV_i,j-1 done)
    uint64_t *p_full = s_full + kNQ;                        // [kNQ]: P_ij in TMEM
    uint64_t *o_done = p_full + kNQ;                        // [kNQ]: last P V product done
    uint64_t *fin_bar = o_done + kNQ;
    uint32_t *tmem_base_s = reinterpret_cast<uint32_t *>(fin_bar + 1);
    volatile int32_t *abort_flag = reinterpret_cast<int32_t *>(fin_bar + 2);
    int32_t *sched = reinterpret_cast<int32_t *>(bars + 32);  // [kSortMaxSeqs + 1]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // launched as a programmatic dependent: the next kernel on the stream may
    // be placed once every CTA of this one has started (it waits for this grid
    // itself); nothing is read before the preceding grid has completed
    grid_dependents_launch();
    grid_dependency_wait();
    // CTA order: sequence-major, the heavy (late) query pairs of a sequence
    // first, its kv heads innermost.  Small batches take their sequences
    // longest prefix first, so the longest CTAs start in the first wave
    // rather than the last (the hardware hands out CTAs in index order);
    // each CTA finds its sequence as the one of prefix-length rank
    // blockIdx.x / units (ties by index).
    const int pairs = p.pairs_per_seq;
    const int units = pairs * p.n_kv_heads;
    const int unit = (int)(blockIdx.x % units);
    const int pair = pairs - 1 - unit / p.n_kv_heads;
    const int kvh = unit % p.n_kv_heads;
    int s = (int)(blockIdx.x / units);
    if (p.n_seqs <= kSortMaxSeqs) {
        if (threadIdx.x < p.n_seqs) sched[threadIdx.x] = __ldg(p.prefix_lens + threadIdx.x);
        __syncthreads();
        if (threadIdx.x < p.n_seqs) {
            const int32_t mine = sched[threadIdx.x];
            int rank = 0;
            for (int t = 0; t < p.n_seqs; ++t) {
                const int32_t o = sched[t];
                rank += (o > mine || (o == mine && t < (int)threadIdx.x)) ? 1 : 0;
            }
            if (rank == s) sched[kSortMaxSeqs] = threadIdx.x;
        }
        __syncthreads();
        s = sched[kSortMaxSeqs];
    }
    const int G = p.group;
    const int pos_per_tile = kTM / G;
    const int p0 = pair * kNQ * pos_per_tile;
    const int p_last = min(p0 + kNQ * pos_per_tile, p.chunk) - 1;
    const int32_t P = __ldg(p.prefix_lens + s);
    const int32_t n_keys = P + p_last + 1;
    const bool bad_len = P < 0 || (int64_t)n_keys > (int64_t)p.max_blocks * p.block_size;
    const int n_kt = bad_len ? 0 : (n_keys + kTN - 1) / kTN;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < NK; ++i) {
            mbar_init(&k_full[i], 2);   // the two K producers
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < NV; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < kNQ; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 4);
            mbar_init(&o_done[i], 1);
        }
        mbar_init(fin_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 9) {
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

    if (warp >= 4 * kNQ) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsIssue) : "memory");
        if (warp != 9 && n_kt > 0) {
            // ===================== TMA producers =====================
            const bool is_v = warp == 11;
            if (warp == 8 && lane == 0) {
                prefetch_tensormap(&q_map);
                mbar_arrive_expect_tx(q_full, kNQ * kQTile);
                for (int i = 0; i < kNQ; ++i)
                    for (int h = 0; h < PANELS; ++h)
                        tma_load_3d(q_s + i * kQTile + h * kQPanel, &q_map, h * 64, kvh * G,
                                    s * p.chunk + p0 + i * pos_per_tile, q_full);
            }
            if (lane == 0) prefetch_tensormap(is_v ? &v_map : &k_map);
            // this warp's 16-key groups: all eight (V) or four (each K warp)
            const int n_grp = is_v ? kTN / 16 : kTN / 32;
            const int grp = is_v ? lane : (warp == 10 ? kTN / 32 : 0) + lane;
            const int NSL = is_v ? NV : NK;
            uint64_t *full = is_v ? v_full : k_full;
            uint64_t *empty = is_v ? v_empty : k_empty;
            uint8_t *ring = is_v ? v_ring : k_ring;
            const uint32_t bytes = is_v ? kSlotBytes : kSlotBytes / 2;
            const int32_t *trow = p.tables + (int64_t)s * p.max_blocks;
            // block ids are read one tile ahead and turned into pool rows when the
            // tile is issued
            auto load_block = [&](int j) -> int32_t {
                const int32_t key0 = j * kTN + grp * 16;
                return (lane < n_grp && key0 < n_keys) ? __ldg(trow + key0 / p.block_size) : 0;
            };
            int32_t blk = load_block(0);
            int issued = 0;
            for (int j = 0; j < n_kt; ++j) {
                int32_t row = p.pool_rows;  // out of range: the box reads zeros
                {
                    const int32_t key0 = j * kTN + grp * 16;
                    if (lane < n_grp && key0 < n_keys) {
                        if (blk < 0 || blk > p.n_blocks)
                            report(p.dev_status, PKV_DEV_BAD_BLOCK_ID);
                        else
                            row = blk * p.block_size + key0 % p.block_size;
                    }
                }
                if (j + 1 < n_kt) blk = load_block(j + 1);
                const int st = j % NSL, use = j / NSL;
                if (lane == 0 && !mbar_wait(&empty[st], (use & 1) ^ 1, abort_flag, p.wait_ns)) {
                    report(p.dev_status, PKV_DEV_TIMEOUT);
                    *abort_flag = 1;
                }
                if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;
                uint8_t *dst = ring + st * kSlotBytes;
                if (lane == 0) mbar_arrive_expect_tx(&full[st], bytes);
                __syncwarp();
                if (lane < n_grp) {
                    if (is_v) {
                        tma_load_3d(dst + grp * kVGroup, &v_map, 0, row, kvh * PANELS, &full[st]);
                    } else {
#pragma unroll
                        for (int h = 0; h < PANELS; ++h)
                            tma_load_3d(dst + h * kKVPanel + grp * 2048, &k_map, h * 64, kvh, row, &full[st]);
                    }
                }
                ++issued;
            }
            // every copy this warp issued has landed before the CTA can exit
            if (lane == 0) {
                if (warp == 8) (void)mbar_wait(q_full, 0);
                for (int i = issued > NSL ? issued - NSL : 0; i < issued; ++i)
                    (void)mbar_wait(&full[i % NSL], (i / NSL) & 1);
            }
        } else if (warp == 9 && n_kt > 0) {
            // ===================== MMA issuer =====================
            const uint32_t idesc_s = umma_idesc_bf16(kTM, kTN, false, false);
            const uint32_t idesc_o = umma_idesc_bf16(kTM, D, false, true);
            bool ok = true;
            if (lane == 0) {
                // The issuing thread bounds the prefill: its waits keep the default
                // limit, which compiles to the plain wait (the settable limit is
                // taken by the producers and the softmax warps; when theirs runs
                // out, the abort flag ends these waits too).
                auto wait_k = [&](int j) { return mbar_wait(&k_full[j % NK], (j / NK) & 1, abort_flag); };
                auto wait_v = [&](int j) { return mbar_wait(&v_full[j % NV], (j / NV) & 1, abort_flag); };
                // S_tj = Q_t K_j^T, then the commit that hands S_tj to warpgroup t
                // Descriptors of a tile are built once and stepped by constants: the
                // start-address field is addr / 16 (14 bits, shared addresses < 256 KiB),
                // so desc(addr + off) = desc(addr) + off / 16 for 16-byte multiples off.
                auto issue_s = [&](int t, int j) {
                    const uint64_t q_desc = umma_desc_sw128(smem_u32(q_s + t * kQTile), 16, 1024);
                    const uint64_t k_desc = umma_desc_sw128(smem_u32(k_ring + (j % NK) * kSlotBytes), 16, 1024);
                    if constexpr (D == 128) {
                        uint64_t ad[8], bd[8];
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            ad[kk] = desc_step(q_desc, (kk / 4) * kQPanel + (kk % 4) * 32);
                            bd[kk] = desc_step(k_desc, (kk / 4) * kKVPanel + (kk % 4) * 32);
                        }
                        umma_bf16_x8(tmem + t * kTileCols, ad, bd, idesc_s, 0u);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)
                            umma_bf16(tmem + t * kTileCols, desc_step(q_desc, (kk / 4) * kQPanel + (kk % 4) * 32),
                                      desc_step(k_desc, (kk / 4) * kKVPanel + (kk % 4) * 32), idesc_s, kk > 0);
                    }
                    umma_commit(&s_full[t]);
                };
                ok = mbar_wait(q_full, 0, abort_flag) && wait_k(0);
                if (ok) {
                    tc_fence_after();
                    for (int t = 0; t < kNQ; ++t) issue_s(t, 0);
                    umma_commit(&k_empty[0]);
                }
                for (int j = 0; ok && j < n_kt; ++j) {
                    ok = wait_v(j);
                    if (!ok) break;
                    const uint64_t v_desc = umma_desc_sw128(smem_u32(v_ring + (j % NV) * kSlotBytes), 2048, 1024);
                    for (int t = 0; t < kNQ && ok; ++t) {
                        ok = mbar_wait(&p_full[t], j & 1, abort_flag);
                        if (!ok) break;
                        tc_fence_after();
                        // O_t += P_tj V_j: A = P (TMEM, 8 columns per 16 keys), B = V (MN-major:
                        // 16-key group kk at kk * kVGroup, its two 8-key halves 1024 B
                        // apart, 64-column panels 2048 B apart)
                        {
                            static_assert(kTN / 16 == 8, "eight 16-key products per tile");
                            uint64_t bd[8];
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) bd[kk] = desc_step(v_desc, kk * kVGroup);
                            umma_bf16_ts_x8(tmem + t * kTileCols + kOCol, tmem + t * kTileCols, bd, idesc_o,
                                            j > 0 ? 1u : 0u);
                        }
                        if (j + 1 < n_kt) {
                            if (t == 0) {
                                ok = wait_k(j + 1);
                                if (!ok) break;
                                tc_fence_after();
                            }
                            issue_s(t, j + 1);
                        } else {
                            umma_commit(&o_done[t]);
                        }
                    }
                    if (!ok) break;
                    umma_commit(&v_empty[j % NV]);
                    if (j + 1 < n_kt) umma_commit(&k_empty[(j + 1) % NK]);
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
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsSoftmax) : "memory");
        // ===================== softmax warpgroups: row r of tile qt = TMEM lane r =====================
        const int qt = warp / 4;
        const int r = threadIdx.x % kTM;
        const int32_t qpos = P + p0 + qt * pos_per_tile + r / G;
        const uint32_t lane_base = tmem + ((uint32_t)((warp % 4) * 32) << 16) + qt * kTileCols;
        float m = -INFINITY, l = 0.f;
        bool ok = n_kt > 0;
        for (int j = 0; j < n_kt && ok; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(&s_full[qt], j & 1, abort_flag, p.wait_ns));
            if (!ok) break;
            tc_fence_after();
            const int32_t key_base = j * kTN;
            // rows whose keys in this tile are all visible need no per-key test
            const bool masked = __any_sync(0xffffffffu, key_base + kTN - 1 > qpos);
            uint32_t sv[kTN];
#pragma unroll
            for (int c = 0; c < kTN / 32; ++c) tmem_ld32_async(lane_base + c * 32, sv + c * 32);
            tmem_wait_ld();
            // keys past this row's position get a score of -inf (exp2 gives 0);
            // only tiles crossing the diagonal take this branch
            if (masked) {
#pragma unroll
                for (int i = 0; i < kTN; ++i)
                    if (key_base + i > qpos) sv[i] = __float_as_uint(-INFINITY);
            }
            // row maximum: three-input max over four independent chains
            float mx;
            {
                float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
                for (int i = 0; i < kTN; i += 8) {
                    a0 = fmax3(a0, __uint_as_float(sv[i]), __uint_as_float(sv[i + 1]));
                    a1 = fmax3(a1, __uint_as_float(sv[i + 2]), __uint_as_float(sv[i + 3]));
                    a2 = fmax3(a2, __uint_as_float(sv[i + 4]), __uint_as_float(sv[i + 5]));
                    a3 = fmax3(a3, __uint_as_float(sv[i + 6]), __uint_as_float(sv[i + 7]));
                }
                mx = fmax3(a0, a1, fmaxf(a2, a3)) * p.scale_log2;
            }
            float alpha = 1.f;
            if (m == -INFINITY) {
                m = mx;          // first tile: key 0 is always visible, so mx is finite
            } else if (mx > m + kRescaleThreshold) {
                alpha = fast_exp2(m - mx);
                m = mx;
            }
            // O row rescale (rare): O holds P V up to tile j - 1, complete since
            // S_j's commit came after it
            if (__any_sync(0xffffffffu, alpha != 1.f) && j > 0) {
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32_async(lane_base + kOCol + c * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                    tmem_st32(lane_base + kOCol + c * 32, v);
                }
            }
            // probabilities (packed two-lane FMA for the exponent arguments) and
            // two packed partial row sums; P (bf16 pairs) over S's first 64
            // columns, each 16-column store after the S columns it covers were read
            const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(-m, -m);
            float2 la = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < kTN / 32; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int kidx = c * 32 + 2 * e;
                    const float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[kidx]), __uint_as_float(sv[kidx + 1])),
                                                sc2, nm2);
                    const float2 ee = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                    if (e & 1)
                        lb = __fadd2_rn(lb, ee);
                    else
                        la = __fadd2_rn(la, ee);
                    pk[e] = pack_bf16x2(ee.x, ee.y);
                }
                tmem_st16_async(lane_base + c * 16, pk);
            }
            l = l * alpha + ((la.x + la.y) + (lb.x + lb.y));
            tmem_wait_st();
            // last tile: V rows of keys past the last one may hold anything; zero
            // them once V_j has landed (both warpgroups write the same zeros)
            if (j == n_kt - 1 && (n_keys & 15) != 0) {
                ok = __all_sync(0xffffffffu, mbar_wait(&v_full[j % NV], (j / NV) & 1, abort_flag, p.wait_ns));
                if (!ok) break;
                const int first = n_keys - key_base, stop = ((n_keys + 15) & ~15) - key_base;
                uint8_t *vs = v_ring + (j % NV) * kSlotBytes;
                for (int i = r; i < (stop - first) * PANELS * 8; i += kTM) {
                    const int row = first + i / (PANELS * 8), pc = i % (PANELS * 8);
                    *reinterpret_cast<uint4 *>(vs + (row / 16) * kVGroup + (pc / 8) * 2048 + swz128(row % 16, pc % 8)) =
                        make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();   // zeroed V rows visible to the tensor core
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[qt]);
        }
        if (ok && n_kt > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(&o_done[qt], 0, abort_flag, p.wait_ns));
            tc_fence_after();
        }
        // the warpgroup agrees before its named barriers (every warp gets here)
        const bool go = wg_and(1 + qt, ok && n_kt > 0);
        if (go) {
            // Row r of O, normalised, into a staging tile laid out like a Q tile
            // ([panel][row][128 B], 128-byte swizzle; the K ring is free: the last S
            // of both tiles retired before either tile's last P V), then one TMA
            // store per panel (positions past the chunk are outside the map).
            const int pos = p0 + qt * pos_per_tile + r / G, h = kvh * G + r % G;
            const float inv = 1.f / l;
            uint8_t *stage = k_ring + qt * kQTile;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tmem_ld32_async(lane_base + kOCol + c * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(v[8 * q4 + 0]) * inv, __uint_as_float(v[8 * q4 + 1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(v[8 * q4 + 2]) * inv, __uint_as_float(v[8 * q4 + 3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(v[8 * q4 + 4]) * inv, __uint_as_float(v[8 * q4 + 5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(v[8 * q4 + 6]) * inv, __uint_as_float(v[8 * q4 + 7]) * inv);
                    const uint32_t chunk = (uint32_t)((c % 2) * 4 + q4);
                    *reinterpret_cast<uint4 *>(stage + (c / 2) * kQPanel + swz128((uint32_t)r, chunk)) = w;
                }
            }
            fence_proxy_async_smem();     // generic writes -> the TMA's reads
            asm volatile("bar.sync %0, 128;" ::"r"(1 + qt) : "memory");
            // a tile whose first position is past the chunk stores nothing; a tile
            // that crosses the chunk's end is clipped by the map
            if (r == 0 && p0 + qt * pos_per_tile <= p_last) {
#pragma unroll
                for (int hp = 0; hp < PANELS; ++hp)
                    tma_store_4d(&o_map, stage + hp * kQPanel, hp * 64, kvh * G, p0 + qt * pos_per_tile, s);
                bulk_wait_read_all();
            }
            if (pos <= p_last && p.lse_out)
                p.lse_out[((int64_t)s * p.chunk + pos) * p.n_q_heads + h] = (m + __log2f(l)) * 0.69314718055994531f;
        } else if (!ok) {
            if (lane == 0) report(p.dev_status, PKV_DEV_TIMEOUT);
            *abort_flag = 1;
        }
    }
    // everyone meets here before the TMEM is released
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t stream)
{
    const pkv_dims &d = a.dims;
    const int G = a.n_q_heads / d.n_kv_heads;
    if (G > 16 || kTM % G != 0) return cudaErrorInvalidValue;
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
    p.wait_ns = pipeline_wait_ns();
    const int pos_per_tile = kTM / G;
    p.tiles_per_seq = (a.chunk + pos_per_tile - 1) / pos_per_tile;
    p.pairs_per_seq = (p.tiles_per_seq + kNQ - 1) / kNQ;
    p.n_seqs = a.n_seqs;
    p.n_kv_heads = d.n_kv_heads;

    CUtensorMap qmap, kmap, vmap, omap;
    {
        const uint64_t dims[3] = {(uint64_t)d.head_dim, (uint64_t)a.n_q_heads, (uint64_t)a.n_seqs * a.chunk};
        const uint64_t strides[2] = {(uint64_t)d.head_dim * 2, (uint64_t)a.n_q_heads * d.head_dim * 2};
        const uint32_t box[3] = {64u, (uint32_t)G, (uint32_t)pos_per_tile};
        if (encode_tensor_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.q), dims, strides,
                              box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // out: {64 columns, query head, chunk position, sequence}; the box of a
        // query tile is the Q box, and positions past the chunk are not written
        const uint64_t dims[4] = {(uint64_t)d.head_dim, (uint64_t)a.n_q_heads, (uint64_t)a.chunk,
                                  (uint64_t)a.n_seqs};
        const uint64_t strides[3] = {(uint64_t)d.head_dim * 2, (uint64_t)a.n_q_heads * d.head_dim * 2,
                                     (uint64_t)a.chunk * a.n_q_heads * d.head_dim * 2};
        const uint32_t box[4] = {64u, (uint32_t)G, (uint32_t)pos_per_tile, 1u};
        if (encode_tensor_map(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, a.out, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const uint64_t rows = (uint64_t)(d.n_blocks + 1) * d.block_size;
    const uint64_t row_bytes = (uint64_t)d.n_kv_heads * d.head_dim * 2;
    {
        // K: {64 columns, kv head, pool row}, one head and 16 rows per box
        const uint64_t dims[3] = {(uint64_t)d.head_dim, (uint64_t)d.n_kv_heads, rows};
        const uint64_t strides[2] = {(uint64_t)d.head_dim * 2, row_bytes};
        const uint32_t box[3] = {64u, 1u, 16u};
        if (encode_tensor_map(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.k_pool), dims, strides,
                              box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        // V: {64 columns, pool row, 64-column panel of all heads}: a box of 16
        // rows and a head's panels lands as [panel][row][128 B]
        const uint32_t panels = (uint32_t)d.head_dim / 64u;
        const uint64_t dims[3] = {64u, rows, (uint64_t)d.n_kv_heads * panels};
        const uint64_t strides[2] = {row_bytes, 128u};
        const uint32_t box[3] = {64u, 16u, panels};
        if (encode_tensor_map(&vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.v_pool), dims, strides,
                              box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }

    const int slots = d.head_dim == 128 ? k_slots<128>() + v_slots<128>() : k_slots<64>() + v_slots<64>();
    const size_t smem = 1024 + (size_t)kNQ * kTM * d.head_dim * 2 + (size_t)slots * kTN * d.head_dim * 2 +
                        32 * sizeof(uint64_t) + (kSortMaxSeqs + 1) * sizeof(int32_t);
    const int64_t ctas = (int64_t)p.pairs_per_seq * d.n_kv_heads * a.n_seqs;
    if (ctas > INT32_MAX) return cudaErrorInvalidValue;
    dim3 grid((unsigned)ctas);
    // The register split assumes the block gets kLaunchRegs per thread: refuse
    // a build whose kernel was given fewer (its setmaxnreg.inc could not complete).
    static const bool regs_ok = [] {
        cudaFuncAttributes fa128{}, fa64{};
        return cudaFuncGetAttributes(&fa128, prefill_tc_kernel<128>) == cudaSuccess &&
               cudaFuncGetAttributes(&fa64, prefill_tc_kernel<64>) == cudaSuccess && fa128.numRegs >= kLaunchRegs &&
               fa64.numRegs >= kLaunchRegs;
    }();
    if (!regs_ok) return cudaErrorInvalidConfiguration;
    // a programmatic dependent of the previous kernel on the stream: its CTAs
    // are placed on SMs as that kernel's CTAs leave them
    cudaLaunchAttribute pdl[1];
    pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pdl[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t lc{};
    lc.gridDim = grid;
    lc.blockDim = dim3(384);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    lc.attrs = pdl;
    lc.numAttrs = 1;
    cudaError_t e;
    if (d.head_dim == 128) {
        e = prepare_kernel(reinterpret_cast<const void *>(prefill_tc_kernel<128>), 384, smem, nullptr);
        if (e != cudaSuccess) return e;
        return cudaLaunchKernelEx(&lc, prefill_tc_kernel<128>, qmap, kmap, vmap, omap, p);
    }
    e = prepare_kernel(reinterpret_cast<const void *>(prefill_tc_kernel<64>), 384, smem, nullptr);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&lc, prefill_tc_kernel<64>, qmap, kmap, vmap, omap, p);
}

}  // namespace pkv
