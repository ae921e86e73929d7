"""GB300-native K-draft verify step for MTP speculative decoding (placeholder)."""
