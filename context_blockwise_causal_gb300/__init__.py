"""GB300-native context-parallel causal attention (placeholder; binding follows)."""
