// launch.h -- internal interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pagedkv.h"

namespace pkv {

struct WriteArgs {
    const void *k_new, *v_new;
    void *k_pool, *v_pool;
    pkv_dims dims;
    const int32_t *tables;
    int32_t max_blocks;
    const int32_t *start_pos;
    int32_t n_seqs, n_new;
    int32_t *dev_status;
};

struct GatherArgs {
    const void *k_pool, *v_pool;
    pkv_dims dims;
    const int32_t *tables;
    int32_t max_blocks;
    const int32_t *lens;
    int32_t n_seqs, out_tokens;
    void *k_out, *v_out;
    int32_t *dev_status;
};

// Decode workspace layout (all offsets 256-byte aligned):
//   header     : uint32 [64]        work counter, items, overflow flag, stages per item, total stages
//   seq_prefix : int32 [n_seqs + 1] 16-token stages before each sequence (balanced mode)
//   seg        : int2  [n_seqs]     (first partial slot, pieces) of each sequence
//   items      : int2  [cap]        fixed splits: (sequence, split) per item; balanced: first sequence
//   part_ml    : float2[cap][Hq]    (running max in log2 units, running sum)
//   part_acc   : float [cap][Hq][D] unnormalised partial outputs
struct DecodeWorkspace {
    uint32_t *header;
    int32_t *seq_prefix;
    int2 *seg;
    int2 *items;
    float2 *part_ml;
    float *part_acc;
    int32_t capacity;  // partial slots (and items) the workspace can hold
};

// Automatic splitting cuts the concatenated token stream into equal pieces,
// about one per CTA; the workspace for it holds n_seqs + this many slots.
constexpr int kDecodeAutoMaxItems = 512;

size_t decode_workspace_bytes(int32_t n_seqs, int32_t n_q_heads, int32_t head_dim,
                              int64_t capacity);
bool carve_decode_workspace(void *ws, size_t bytes, int32_t n_seqs, int32_t n_q_heads,
                            int32_t head_dim, DecodeWorkspace *out);

struct DecodeArgs {
    const void *q;
    int32_t n_q_heads;
    const void *k_pool, *v_pool;
    const float *k_scales, *v_scales;
    int32_t kv_dtype;
    pkv_dims dims;
    const int32_t *tables;
    int32_t max_blocks;
    const int32_t *ctx_lens;
    int32_t n_seqs;
    float softmax_scale;
    int32_t split_tokens;  // 0: balanced pieces
    void *out;
    float *lse_out;
    DecodeWorkspace ws;
    int32_t *dev_status;
    float *write_k_scales, *write_v_scales;  // int8 pools of a fused decode step
};

struct PrefillArgs {
    const void *q;
    int32_t n_q_heads;
    const void *k_pool, *v_pool;
    pkv_dims dims;
    const int32_t *tables;
    int32_t max_blocks;
    const int32_t *prefix_lens;
    int32_t n_seqs, chunk;
    float softmax_scale;
    void *out;
    float *lse_out;
    int32_t *dev_status;
};

cudaError_t launch_write_bf16(const WriteArgs &a, cudaStream_t stream);
cudaError_t launch_write_int8(const WriteArgs &a, float *k_scales, float *v_scales,
                              cudaStream_t stream);
cudaError_t launch_gather(const GatherArgs &a, int num_sms, cudaStream_t stream);
cudaError_t launch_copy_blocks(const int32_t *pairs, int32_t n_pairs, void *k_pool, void *v_pool, float *k_scales,
                               float *v_scales, bool int8, const pkv_dims &d, int32_t *dev_status, int num_sms,
                               cudaStream_t stream);
// write (nullable): this step's new rows, written by the first launch of the
// decode (the fused decode step).
cudaError_t launch_decode(const DecodeArgs &a, int num_sms, cudaStream_t stream, const WriteArgs *write = nullptr);
cudaError_t launch_prefill(const PrefillArgs &a, int num_sms, cudaStream_t stream);

// The limit in nanoseconds of the kernels' pipeline waits (default 4 s; see
// pkv_set_pipeline_wait_ns in pagedkv.h), read when a launch is prepared.
unsigned long long pipeline_wait_ns();

// Driver entry point for tensor-map encoding (resolved once through cudart,
// so the library does not link libcuda directly).  Returns CUDA_SUCCESS or
// the driver error.  Maps of recent calls with the same arguments are reused.
CUresult encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, uint32_t rank,
                           void *base, const uint64_t *dims, const uint64_t *strides_bytes,
                           const uint32_t *box, CUtensorMapSwizzle swizzle);

// Before a launch of `kern` with `smem` bytes of dynamic shared memory on the
// current device: raises the kernel's dynamic shared memory limit when smem
// exceeds what was set before (it never lowers it) and, if occupancy is not
// null, returns the resident CTAs per SM at (threads, smem).  Both are done
// once per kernel, device and combination.
cudaError_t prepare_kernel(const void *kern, int threads, size_t smem, int *occupancy);

}  // namespace pkv
