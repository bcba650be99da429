"""GB300-native Super Bloom filter (placeholder during bring-up)."""
