"""GB300-native HSTU jagged attention (sm_103a CUDA behind a C ABI)."""
