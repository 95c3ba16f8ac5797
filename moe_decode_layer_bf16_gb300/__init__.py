"""GB300-native MoE decode layer (placeholder; the binding is added next)."""
