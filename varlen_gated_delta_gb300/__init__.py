"""GB300-native packed variable-length gated-delta layer (placeholder; binding lands next)."""
