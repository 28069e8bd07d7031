"""GB300-native RMSNorm forward/backward (placeholder; binding added next)."""
