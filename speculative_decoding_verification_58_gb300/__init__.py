"""GB300-native batched speculative-decoding verification (placeholder; binding added with the C-ABI)."""
