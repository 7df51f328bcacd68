"""GB300-native FAST-AR per-chunk attention step (TempCache + AnnSA + AnnCA)."""
