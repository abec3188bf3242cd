"""GB300-native lightning attention (chunkwise decayed causal linear attention)."""
