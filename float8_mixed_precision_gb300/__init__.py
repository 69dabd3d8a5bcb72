"""GB300-native Float8 training linear with dynamic tensorwise scaling."""
