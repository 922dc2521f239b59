"""GB300-native prefill context-parallel causal attention (zigzag / interleave + LSE merge)."""
