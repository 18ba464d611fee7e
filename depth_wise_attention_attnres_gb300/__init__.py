"""GB300-native AttnRes depth-wise aggregation (Full and Block AttnRes)."""
