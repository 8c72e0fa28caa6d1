// api.cu -- the extern "C" entry points of libpagedkv.so: argument checks on
// the host, then kernel launches on the caller's stream.  No allocation, no
// synchronisation, no exception crosses the ABI.
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "decode_small.h"

namespace pkv {

cudaError_t launch_prefill_tc(const PrefillArgs &a, cudaStream_t stream);

namespace {

thread_local int g_last_cuda_error = 0;
std::atomic<uint64_t> g_pipeline_wait_ns{kWaitTimeoutNs};

int cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return PKV_OK;
    g_last_cuda_error = (int)e;
    return PKV_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int num_sms_of_current_device(int *out)
{
    static int cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev >= 0 && dev < 64 && cache[dev] > 0) {
        *out = cache[dev];
        return PKV_OK;
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev >= 0 && dev < 64) cache[dev] = n;
    *out = n;
    return PKV_OK;
}

// Geometry every kernel supports: head_dim 64 or 128, block_size a multiple of
// 16 up to 256, at least one kv head, a non-negative block count.
int check_dims(const pkv_dims &d)
{
    if (d.n_blocks < 0 || d.block_size <= 0 || d.n_kv_heads <= 0 || d.head_dim <= 0)
        return PKV_ERR_INVALID_ARG;
    if (d.head_dim != 64 && d.head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (d.block_size % 16 != 0 || d.block_size > 256) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)(d.n_blocks + 1) * d.block_size > 0x7fffffffLL) return PKV_ERR_OUT_OF_RANGE;
    return PKV_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Partial slots a call needs: fixed splits give one per split of every
// sequence; balanced pieces give at most one per sequence plus one per item.
size_t decode_capacity_for(int32_t n_seqs, int64_t max_total_ctx_tokens, int32_t split_tokens)
{
    if (split_tokens > 0) return (size_t)((max_total_ctx_tokens + split_tokens - 1) / split_tokens + n_seqs);
    const int64_t stages = (max_total_ctx_tokens + 15) / 16 + 1;
    return (size_t)(n_seqs + (stages < kDecodeAutoMaxItems ? stages : kDecodeAutoMaxItems));
}

}  // namespace

void record_cuda_error(int e) { g_last_cuda_error = e; }

unsigned long long pipeline_wait_ns() { return g_pipeline_wait_ns.load(); }

namespace {

// A tensor map depends only on its arguments, so the maps of recent calls are
// kept and a call whose arguments match one reuses it (a model's pools give
// the same few maps at every step); the key is zero-filled so that whole keys
// compare byte for byte.
struct MapKey {
    const void *base;
    uint64_t dims[5];
    uint64_t strides[4];
    uint32_t box[5];
    int32_t dtype, rank, swizzle, pad;
};
struct MapEntry {
    MapKey key;
    CUtensorMap map;
    bool used;
};
constexpr int kMapCacheEntries = 32;
MapEntry g_maps[kMapCacheEntries];
int g_map_next = 0;
std::mutex g_map_mu;

// Per kernel and device: the largest dynamic shared memory size set so far (the
// attribute only grows, so every earlier size stays launchable) and the
// occupancy of the (threads, smem) combinations seen.
struct KernelEntry {
    const void *kern;
    int device, threads;
    size_t smem, smem_set;
    int occupancy;
};
constexpr int kKernelCacheEntries = 64;
KernelEntry g_kernels[kKernelCacheEntries];
int g_kernels_used = 0;
std::mutex g_kernel_mu;

}  // namespace

CUresult encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, uint32_t rank, void *base,
                           const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                           CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return CUDA_ERROR_NOT_FOUND;
    if (rank < 1 || rank > 5) return CUDA_ERROR_INVALID_VALUE;
    MapKey key;
    memset(&key, 0, sizeof key);
    key.base = base;
    for (uint32_t i = 0; i < rank; ++i) {
        key.dims[i] = dims[i];
        key.box[i] = box[i];
        if (i + 1 < rank) key.strides[i] = strides_bytes[i];
    }
    key.dtype = (int32_t)dtype;
    key.rank = (int32_t)rank;
    key.swizzle = (int32_t)swizzle;
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        for (const MapEntry &e : g_maps)
            if (e.used && memcmp(&e.key, &key, sizeof key) == 0) {
                *map = e.map;
                return CUDA_SUCCESS;
            }
    }
    cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
    const CUresult r = fn(map, dtype, rank, base, reinterpret_cast<const cuuint64_t *>(dims),
                          reinterpret_cast<const cuuint64_t *>(strides_bytes), reinterpret_cast<const cuuint32_t *>(box),
                          elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS) {
        std::lock_guard<std::mutex> lock(g_map_mu);
        MapEntry &e = g_maps[g_map_next];
        g_map_next = (g_map_next + 1) % kMapCacheEntries;
        e.key = key;
        e.map = *map;
        e.used = true;
    }
    return r;
}

cudaError_t prepare_kernel(const void *kern, int threads, size_t smem, int *occupancy)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(g_kernel_mu);
    size_t smem_set = 0;
    for (int i = 0; i < g_kernels_used; ++i) {
        const KernelEntry &e = g_kernels[i];
        if (e.kern != kern || e.device != dev) continue;
        if (e.smem_set > smem_set) smem_set = e.smem_set;
        if (e.threads == threads && e.smem == smem && (occupancy == nullptr || e.occupancy >= 0)) {
            if (occupancy) *occupancy = e.occupancy;
            return cudaSuccess;
        }
    }
    if (smem > smem_set) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        smem_set = smem;
    }
    int occ = -1;
    if (occupancy) {
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem);
        if (err != cudaSuccess) return err;
        *occupancy = occ;
    }
    // remember the combination, and the size now set, for every entry of this kernel and device
    for (int i = 0; i < g_kernels_used; ++i)
        if (g_kernels[i].kern == kern && g_kernels[i].device == dev) g_kernels[i].smem_set = smem_set;
    if (g_kernels_used < kKernelCacheEntries)
        g_kernels[g_kernels_used++] = KernelEntry{kern, dev, threads, smem, smem_set, occ};
    return cudaSuccess;
}

// Prefill runs on the tcgen05 kernel (prefill_tc.cu).
cudaError_t launch_prefill(const PrefillArgs &a, int num_sms, cudaStream_t stream)
{
    (void)num_sms;
    return launch_prefill_tc(a, stream);
}

}  // namespace pkv

using namespace pkv;

extern "C" {

const char *pkv_status_string(int status)
{
    switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_OUT_OF_RANGE: return "PKV_ERR_OUT_OF_RANGE";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    case PKV_ERR_OUT_OF_BLOCKS: return "PKV_ERR_OUT_OF_BLOCKS";
    case PKV_ERR_STATE: return "PKV_ERR_STATE";
    default: return "PKV_ERR_UNKNOWN";
    }
}

int pkv_last_cuda_error(void) { return g_last_cuda_error; }

uint64_t pkv_set_pipeline_wait_ns(uint64_t ns)
{
    const uint64_t prev = g_pipeline_wait_ns.exchange(ns == 0 ? (uint64_t)kWaitTimeoutNs : ns);
    return prev;
}

static int write_common_checks(const void *k_new, const void *v_new, const void *k_pool, const void *v_pool,
                               const pkv_dims &dims, const int32_t *tables, int32_t max_blocks,
                               const int32_t *start_pos, int32_t n_seqs, int32_t n_new)
{
    int st = check_dims(dims);
    if (st != PKV_OK) return st;
    if (n_seqs < 0 || n_new < 0 || max_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (n_seqs == 0 || n_new == 0) return PKV_OK;
    if (!k_new || !v_new || !k_pool || !v_pool || !tables || !start_pos) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
        return PKV_ERR_INVALID_ARG;
    if ((int64_t)n_new > (int64_t)max_blocks * dims.block_size) return PKV_ERR_OUT_OF_RANGE;
    return PKV_OK;
}

int paged_kv_write(const pkv_bf16 *k_new, const pkv_bf16 *v_new, pkv_bf16 *k_pool, pkv_bf16 *v_pool,
                   pkv_dims dims, const int32_t *block_tables, int32_t max_blocks, const int32_t *start_pos,
                   int32_t n_seqs, int32_t n_new, int32_t *dev_status, pkv_stream_t stream)
{
    int st = write_common_checks(k_new, v_new, k_pool, v_pool, dims, block_tables, max_blocks, start_pos,
                                 n_seqs, n_new);
    if (st != PKV_OK || n_seqs == 0 || n_new == 0) return st;
    WriteArgs a{k_new, v_new, k_pool, v_pool, dims, block_tables, max_blocks, start_pos, n_seqs, n_new,
                dev_status};
    return cuda_status(launch_write_bf16(a, (cudaStream_t)stream));
}

int paged_kv_write_int8(const pkv_bf16 *k_new, const pkv_bf16 *v_new, int8_t *k_pool, int8_t *v_pool,
                        float *k_scales, float *v_scales, pkv_dims dims, const int32_t *block_tables,
                        int32_t max_blocks, const int32_t *start_pos, int32_t n_seqs, int32_t n_new,
                        int32_t *dev_status, pkv_stream_t stream)
{
    int st = write_common_checks(k_new, v_new, k_pool, v_pool, dims, block_tables, max_blocks, start_pos,
                                 n_seqs, n_new);
    if (st != PKV_OK || n_seqs == 0 || n_new == 0) return st;
    if (!k_scales || !v_scales) return PKV_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k_scales) | reinterpret_cast<uintptr_t>(v_scales)) & 3u)
        return PKV_ERR_INVALID_ARG;
    WriteArgs a{k_new, v_new, k_pool, v_pool, dims, block_tables, max_blocks, start_pos, n_seqs, n_new,
                dev_status};
    return cuda_status(launch_write_int8(a, k_scales, v_scales, (cudaStream_t)stream));
}

int paged_kv_gather(const pkv_bf16 *k_pool, const pkv_bf16 *v_pool, pkv_dims dims, const int32_t *block_tables,
                    int32_t max_blocks, const int32_t *lens, int32_t n_seqs, int32_t out_tokens,
                    pkv_bf16 *k_out, pkv_bf16 *v_out, int32_t *dev_status, pkv_stream_t stream)
{
    int st = check_dims(dims);
    if (st != PKV_OK) return st;
    if (n_seqs < 0 || out_tokens < 0 || max_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (n_seqs == 0 || out_tokens == 0) return PKV_OK;
    if (!k_pool || !v_pool || !block_tables || !lens || !k_out || !v_out) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_out) || !aligned16(v_out))
        return PKV_ERR_INVALID_ARG;
    int sms = 0;
    st = num_sms_of_current_device(&sms);
    if (st != PKV_OK) return st;
    GatherArgs a{k_pool, v_pool, dims, block_tables, max_blocks, lens, n_seqs, out_tokens, k_out, v_out,
                 dev_status};
    return cuda_status(launch_gather(a, sms, (cudaStream_t)stream));
}

int paged_kv_copy_blocks(const int32_t *pairs, int32_t n_pairs, void *k_pool, void *v_pool, float *k_scales,
                         float *v_scales, int32_t kv_dtype, pkv_dims dims, int32_t *dev_status,
                         pkv_stream_t stream)
{
    int st = check_dims(dims);
    if (st != PKV_OK) return st;
    if (n_pairs < 0) return PKV_ERR_INVALID_ARG;
    if (kv_dtype != PKV_KV_BF16 && kv_dtype != PKV_KV_INT8) return PKV_ERR_UNSUPPORTED;
    if (n_pairs == 0) return PKV_OK;
    if (!pairs || !k_pool || !v_pool || !aligned16(k_pool) || !aligned16(v_pool)) return PKV_ERR_INVALID_ARG;
    const bool int8 = kv_dtype == PKV_KV_INT8;
    if (int8 && (!k_scales || !v_scales || !aligned16(k_scales) || !aligned16(v_scales)))
        return PKV_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(pairs) % 8 != 0) return PKV_ERR_INVALID_ARG;
    int sms = 0;
    st = num_sms_of_current_device(&sms);
    if (st != PKV_OK) return st;
    return cuda_status(launch_copy_blocks(pairs, n_pairs, k_pool, v_pool, k_scales, v_scales, int8, dims,
                                          dev_status, sms, (cudaStream_t)stream));
}

size_t pkv_decode_workspace_bytes(int32_t n_seqs, int32_t n_q_heads, int32_t head_dim,
                                  int64_t max_total_ctx_tokens, int32_t split_tokens)
{
    if (n_seqs < 0 || n_q_heads <= 0 || head_dim <= 0 || max_total_ctx_tokens < 0 || split_tokens < 0 ||
        (split_tokens > 0 && split_tokens % 16 != 0))
        return 0;
    // no sequence attends more than INT32_MAX tokens: a larger bound is an
    // error (and keeps the slot arithmetic below far from overflow)
    if (max_total_ctx_tokens > (int64_t)n_seqs * 0x7fffffffLL) return 0;
    return decode_workspace_bytes(n_seqs, n_q_heads, head_dim,
                                  (int64_t)decode_capacity_for(n_seqs, max_total_ctx_tokens, split_tokens));
}

// Small batches (one wave of (sequence, kv head) units, short contexts, bf16
// pages, automatic splitting) take the one-launch path of decode_small.cu;
// PKV_DECODE_IMPL=split in the environment keeps every call on the split-KV
// path (for comparisons).
static bool use_small_decode(const DecodeArgs &a, int sms)
{
    const char *impl = getenv("PKV_DECODE_IMPL");
    if (impl && strcmp(impl, "split") == 0) return false;
    return decode_small_eligible(a, sms);
}

// Host checks of a decode call; on success fills *a (workspace carved).
static int prepare_decode(const pkv_bf16 *q, int32_t n_q_heads, const void *k_pool, const void *v_pool,
                          const float *k_scales, const float *v_scales, int32_t kv_dtype, const pkv_dims &dims,
                          const int32_t *block_tables, int32_t max_blocks, const int32_t *ctx_lens, int32_t n_seqs,
                          float softmax_scale, int32_t split_tokens, pkv_bf16 *out, float *lse_out,
                          void *workspace, size_t workspace_bytes, int32_t *dev_status, DecodeArgs *a)
{
    int st = check_dims(dims);
    if (st != PKV_OK) return st;
    if (n_seqs < 0 || n_q_heads <= 0 || max_blocks <= 0 || split_tokens < 0) return PKV_ERR_INVALID_ARG;
    if (n_q_heads % dims.n_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    const int G = n_q_heads / dims.n_kv_heads;
    if (G > 8 || (G & (G - 1)) != 0) return PKV_ERR_UNSUPPORTED;
    if (kv_dtype != PKV_KV_BF16 && kv_dtype != PKV_KV_INT8) return PKV_ERR_UNSUPPORTED;
    if (split_tokens % 16 != 0) return PKV_ERR_UNSUPPORTED;
    if ((int64_t)max_blocks * dims.block_size > 0x7fffffffLL) return PKV_ERR_OUT_OF_RANGE;
    if (kv_dtype == PKV_KV_INT8 && (dims.n_kv_heads % 4 != 0)) return PKV_ERR_UNSUPPORTED;
    if (n_seqs == 0) return PKV_OK;
    if (!q || !k_pool || !v_pool || !block_tables || !ctx_lens || !out) return PKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out)) return PKV_ERR_INVALID_ARG;
    if (kv_dtype == PKV_KV_INT8 && (!k_scales || !v_scales || !aligned16(k_scales) || !aligned16(v_scales)))
        return PKV_ERR_INVALID_ARG;
    if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f)) return PKV_ERR_INVALID_ARG;
    if (!carve_decode_workspace(workspace, workspace_bytes, n_seqs, n_q_heads, dims.head_dim, &a->ws))
        return PKV_ERR_WORKSPACE;
    a->q = q;
    a->n_q_heads = n_q_heads;
    a->k_pool = k_pool;
    a->v_pool = v_pool;
    a->k_scales = k_scales;
    a->v_scales = v_scales;
    a->kv_dtype = kv_dtype;
    a->dims = dims;
    a->tables = block_tables;
    a->max_blocks = max_blocks;
    a->ctx_lens = ctx_lens;
    a->n_seqs = n_seqs;
    a->softmax_scale = softmax_scale;
    a->split_tokens = split_tokens;
    a->out = out;
    a->lse_out = lse_out;
    a->dev_status = dev_status;
    return PKV_OK;
}

int paged_decode_attention(const pkv_bf16 *q, int32_t n_q_heads, const void *k_pool, const void *v_pool,
                           const float *k_scales, const float *v_scales, int32_t kv_dtype, pkv_dims dims,
                           const int32_t *block_tables, int32_t max_blocks, const int32_t *ctx_lens,
                           int32_t n_seqs, float softmax_scale, int32_t split_tokens, pkv_bf16 *out,
                           float *lse_out, void *workspace, size_t workspace_bytes, int32_t *dev_status,
                           pkv_stream_t stream)
{
    DecodeArgs a{};
    int st = prepare_decode(q, n_q_heads, k_pool, v_pool, k_scales, v_scales, kv_dtype, dims, block_tables,
                            max_blocks, ctx_lens, n_seqs, softmax_scale, split_tokens, out, lse_out, workspace,
                            workspace_bytes, dev_status, &a);
    if (st != PKV_OK || n_seqs == 0) return st;
    int sms = 0;
    st = num_sms_of_current_device(&sms);
    if (st != PKV_OK) return st;
    if (use_small_decode(a, sms)) return cuda_status(launch_decode_small(a, nullptr, (cudaStream_t)stream));
    return cuda_status(launch_decode(a, sms, (cudaStream_t)stream));
}

int paged_decode_step(const pkv_bf16 *k_new, const pkv_bf16 *v_new, const int32_t *start_pos, int32_t n_new,
                      const pkv_bf16 *q, int32_t n_q_heads, void *k_pool, void *v_pool, float *k_scales,
                      float *v_scales, int32_t kv_dtype, pkv_dims dims, const int32_t *block_tables,
                      int32_t max_blocks, const int32_t *ctx_lens, int32_t n_seqs, float softmax_scale,
                      int32_t split_tokens, pkv_bf16 *out, float *lse_out, void *workspace,
                      size_t workspace_bytes, int32_t *dev_status, pkv_stream_t stream)
{
    int st = write_common_checks(k_new, v_new, k_pool, v_pool, dims, block_tables, max_blocks, start_pos, n_seqs,
                                 n_new);
    if (st != PKV_OK) return st;
    DecodeArgs a{};
    st = prepare_decode(q, n_q_heads, k_pool, v_pool, k_scales, v_scales, kv_dtype, dims, block_tables, max_blocks,
                        ctx_lens, n_seqs, softmax_scale, split_tokens, out, lse_out, workspace, workspace_bytes,
                        dev_status, &a);
    if (st != PKV_OK || n_seqs == 0) return st;
    a.write_k_scales = k_scales;
    a.write_v_scales = v_scales;
    WriteArgs w{k_new, v_new, k_pool, v_pool, dims, block_tables, max_blocks, start_pos, n_seqs, n_new, dev_status};
    int sms = 0;
    st = num_sms_of_current_device(&sms);
    if (st != PKV_OK) return st;
    if (use_small_decode(a, sms)) return cuda_status(launch_decode_small(a, &w, (cudaStream_t)stream));
    return cuda_status(launch_decode(a, sms, (cudaStream_t)stream, &w));
}

int paged_prefill_attention(const pkv_bf16 *q, int32_t n_q_heads, const pkv_bf16 *k_pool, const pkv_bf16 *v_pool,
                            pkv_dims dims, const int32_t *block_tables, int32_t max_blocks,
                            const int32_t *prefix_lens, int32_t n_seqs, int32_t chunk, float softmax_scale,
                            pkv_bf16 *out, float *lse_out, int32_t *dev_status, pkv_stream_t stream)
{
    int st = check_dims(dims);
    if (st != PKV_OK) return st;
    if (n_seqs < 0 || chunk < 0 || n_q_heads <= 0 || max_blocks <= 0) return PKV_ERR_INVALID_ARG;
    if (n_q_heads % dims.n_kv_heads != 0) return PKV_ERR_INVALID_ARG;
    const int G = n_q_heads / dims.n_kv_heads;
    if (G > 16 || 64 % G != 0) return PKV_ERR_UNSUPPORTED;
    if (n_seqs == 0 || chunk == 0) return PKV_OK;
    if ((int64_t)chunk > (int64_t)max_blocks * dims.block_size) return PKV_ERR_OUT_OF_RANGE;
    if ((int64_t)n_seqs * chunk > 0x7fffffffLL) return PKV_ERR_OUT_OF_RANGE;
    if (!q || !k_pool || !v_pool || !block_tables || !prefix_lens || !out) return PKV_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out)) return PKV_ERR_INVALID_ARG;
    if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f)) return PKV_ERR_INVALID_ARG;
    int sms = 0;
    st = num_sms_of_current_device(&sms);
    if (st != PKV_OK) return st;
    PrefillArgs a{q, n_q_heads, k_pool, v_pool, dims, block_tables, max_blocks, prefix_lens, n_seqs, chunk,
                  softmax_scale, out, lse_out, dev_status};
    return cuda_status(launch_prefill(a, sms, (cudaStream_t)stream));
}

}  // extern "C"
