"""GB300-native cross-token gate aggregation (TANGO / WANGO)."""
