"""GB300-native batched decode attention over a paged KV cache."""
