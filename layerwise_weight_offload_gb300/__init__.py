"""GB300-native per-block weight stream of Distributed Layerwise Offload.

``dlo`` is the ctypes binding of the C ABI in ``include/dlo.h``; ``stack``
assembles a streamed (two-slot) or all-resident block stack from it;
``workloads`` names the synthetic workloads and seeds their inputs.
"""
