// decode_small.h -- the one-launch decode step for small batches (internal).
#pragma once

#include "launch.h"

namespace pkv {

// The one-launch path holds a head's whole context (K and V rows) in shared
// memory: at most kSmallKVBytes of them, i.e. max_blocks * block_size of at
// most 256 tokens at head_dim 128 and 512 at head_dim 64.
constexpr int kSmallKVBytes = 128 * 1024;
constexpr int kSmallMaxBlocks = 512 / 16;   // table entries of the longest context (block_size >= 16)
int small_max_tokens(int head_dim);

// bf16 pages, automatic splitting, at most one (sequence, kv head) unit per SM
// and contexts that fit the shared-memory buffers.
bool decode_small_eligible(const DecodeArgs &a, int num_sms);

// One CTA per (sequence, kv head): the step's rows of that head (write,
// nullable), then the attention of its G query heads over the whole context.
cudaError_t launch_decode_small(const DecodeArgs &a, const WriteArgs *write, cudaStream_t stream);

}  // namespace pkv
