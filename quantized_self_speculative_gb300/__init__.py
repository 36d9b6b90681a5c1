"""GB300-native hot path of quantized self-speculative decoding.

The compute lives in `libnq.so` (hand-written CUDA for sm_103a behind a C ABI,
declared in include/nq.h).  `quantized_self_speculative_gb300.nq` is the thin
ctypes binding; `synth` draws seeded synthetic inputs.
"""
