"""GB300-native all-reduce, reduce-scatter and all-gather over N virtual ranks."""
