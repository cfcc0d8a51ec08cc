"""GB300-native (sm_103a) fused attention forward."""
