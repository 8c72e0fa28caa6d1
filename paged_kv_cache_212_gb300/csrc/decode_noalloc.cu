// decode_noalloc.cu -- paged_decode_attention for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they run decode attention: a plugin whose host framework owns every
// device byte and hands out only inputs and outputs, an embedded or real-time
// runtime with a fixed memory budget decided at start-up, or a loop that must
// not trigger an allocator's implicit synchronisation.  This entry point needs
// no caller workspace: the split-KV scratch (work list, per-split partials) is
// a fixed-size array in this library's own device memory, reserved when the
// library is loaded onto a GPU and held until the process exits.
//
// The existing kernels run unchanged; only the scratch pointer differs.
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace pkv {
namespace {

// The scratch every call of paged_decode_attention_noalloc uses (16 MiB per
// GPU that loads the library).
constexpr size_t kNoAllocScratchBytes = (size_t)PKV_NOALLOC_DECODE_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_decode_scratch[kNoAllocScratchBytes];

// Device address of g_decode_scratch per device ordinal.  In host code the
// array's name is only a host-side stand-in, so the real address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
// The address is kept for the life of the process: a cudaDeviceReset (or
// anything else that destroys the device's primary context) after the first
// call is not supported, since the array may then live at another address.
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices];

cudaError_t scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        if (!p) return cudaErrorInvalidSymbol;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

void record_cuda_error(int e);  // api.cu: the value pkv_last_cuda_error() reports

}  // namespace pkv

using namespace pkv;

extern "C" int paged_decode_attention_noalloc(const pkv_bf16 *q, int32_t n_q_heads, const void *k_pool,
                                              const void *v_pool, const float *k_scales, const float *v_scales,
                                              int32_t kv_dtype, pkv_dims dims, const int32_t *block_tables,
                                              int32_t max_blocks, const int32_t *ctx_lens, int32_t n_seqs,
                                              float softmax_scale, int32_t split_tokens,
                                              int64_t max_total_ctx_tokens, pkv_bf16 *out, float *lse_out,
                                              int32_t *dev_status, pkv_stream_t stream)
{
    if (n_seqs < 0 || n_q_heads <= 0 || dims.head_dim <= 0 || max_total_ctx_tokens < 0 || split_tokens < 0 ||
        max_total_ctx_tokens > (int64_t)n_seqs * 0x7fffffffLL)
        return PKV_ERR_INVALID_ARG;
    if (n_seqs == 0) return PKV_OK;
    // Reject requests whose scratch would not fit in the static array.
    const size_t need = pkv_decode_workspace_bytes(n_seqs, n_q_heads, dims.head_dim, max_total_ctx_tokens,
                                                   split_tokens);
    if (need == 0) return PKV_ERR_INVALID_ARG;
    if (need > kNoAllocScratchBytes) return PKV_ERR_WORKSPACE;
    void *scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        record_cuda_error((int)e);
        return PKV_ERR_CUDA;
    }
    // Nothing in the scratch has to start at zero: the plan kernel of every
    // call rewrites the work counter, the split count and the work list before
    // anything reads them.  The whole array is handed over, so the work list
    // can hold as many splits as fit.
    return paged_decode_attention(q, n_q_heads, k_pool, v_pool, k_scales, v_scales, kv_dtype, dims, block_tables,
                                  max_blocks, ctx_lens, n_seqs, softmax_scale, split_tokens, out, lse_out, scratch,
                                  kNoAllocScratchBytes, dev_status, stream);
}
