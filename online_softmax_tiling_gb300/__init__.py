"""GB300-native fused attention forward (online-softmax tiling)."""
