"""GB300-native Depth-Staggered Fibonacci Spacing sparse attention."""
