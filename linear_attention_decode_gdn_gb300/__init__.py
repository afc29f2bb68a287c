"""GB300-native batched Gated-DeltaNet decode (dense and DeltaLog append-merge)."""
