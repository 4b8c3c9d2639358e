"""GB300-native tiled online-softmax attention forward (sm_103a)."""
