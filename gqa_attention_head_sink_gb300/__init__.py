"""GB300-native grouped-query attention with a per-head attention sink."""
