"""GB300-native physical-frame state-moments operator (forward + recompute backward)."""
