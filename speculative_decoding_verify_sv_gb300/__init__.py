"""GB300-native verify step of speculative decoding (tree attention + acceptance)."""
