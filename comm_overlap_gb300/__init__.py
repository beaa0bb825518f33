"""GB300-native chunked tensor-parallel MLP (Domino-style row/column splits)."""
