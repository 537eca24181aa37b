"""GB300-native MoE-layer prefill (routed expert FFN, top-k routing, arena
paging). The compute runs in libestream.so (see ``estream``); importing the
package does not load it, so the seeded workload generators stay usable on
machines without the built library."""

__all__ = ["estream", "workloads", "layer", "build"]
