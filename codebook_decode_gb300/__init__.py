"""GB300-native lockstep multi-codebook codec-frame decode (Qwen3-TTS style).

The product is libqtts.so (C ABI in include/qtts.h, CUDA kernels in csrc/);
`qtts` is its ctypes binding and `engine` a thin host-side helper that sets a
model up from named weights and runs frames through that binding.
"""
