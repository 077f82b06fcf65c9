"""GB300-native per-block weight stream of Distributed Layerwise Offload."""
