"""GB300-native rotated-Adam matrix-optimizer step."""
