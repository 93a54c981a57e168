"""GB300-native quantized paged KV cache: quantize-on-write append, paged
split-K decode attention and extend attention (CUDA for sm_103a behind a C ABI)."""
