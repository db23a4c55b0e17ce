"""GB300-native absorbed causal Gated MLA (placeholder; binding follows)."""
