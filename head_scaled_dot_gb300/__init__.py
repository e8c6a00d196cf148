"""GB300-native multi-head attention forward pass.

The compute path is the CUDA library built from ``csrc/`` (C ABI declared in
``include/mha.h``); :mod:`head_scaled_dot_gb300.mha` is its thin Python
binding. Importing this package does not load the library: the binding loads
it on first use and raises if it is missing.
"""

__all__ = ["mha", "workloads", "workcount"]
