"""GB300-native fused MLA attention prolog (sm_103a CUDA behind a C ABI)."""
