"""B300-native DeepSeekMoE layer forward with auxiliary-loss-free routing and
fine-grained FP8 expert GEMMs (CUDA kernels for sm_103a behind a C ABI)."""
