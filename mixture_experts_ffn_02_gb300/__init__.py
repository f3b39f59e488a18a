"""GB300-native sparse MoE feed-forward layer (sm_103a CUDA behind a C ABI)."""
