"""GB300-native GEMV c = B @ a (binding added with the C-ABI library)."""
