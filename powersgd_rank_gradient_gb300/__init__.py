"""GB300-native PowerSGD communication-hook step (CUDA kernels behind a C ABI)."""
