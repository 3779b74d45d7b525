"""GB300-native MoE expert-parallel layout / dispatch / combine and
variable-size reduce-scatterv / all-gatherv (sm_103a CUDA behind a C ABI)."""
