"""FP32 matrix product C = A x B on one GB300 (sm_103a), hand-written CUDA kernels."""
