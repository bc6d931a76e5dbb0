"""GB300-native Ulysses DiT attention (placeholder; the binding lands with the C-ABI)."""
