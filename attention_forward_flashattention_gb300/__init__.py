"""GB300-native fused attention forward (placeholder until the binding lands)."""
