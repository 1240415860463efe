"""GB300-native local Mixture-of-Experts FFN forward (placeholder binding)."""
