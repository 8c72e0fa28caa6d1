"""GB300-native paged KV cache: page write (bf16 / int8), gather, in-place paged
decode attention with split-KV, and chunked paged prefill, as hand-written
sm_103a CUDA kernels behind a C ABI (libpagedkv.so)."""
