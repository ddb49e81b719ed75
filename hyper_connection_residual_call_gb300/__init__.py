"""GB300-native hyper-connection residual call (sm_103a CUDA kernels behind a C ABI)."""
