"""GB300-native W4A16 routed-expert MoE layer.

The layer runs as hand-written CUDA kernels for sm_103a inside
``libmoe_w4a16.so`` behind a C ABI (``include/moe_layer.h``); ``capi`` is the
thin ctypes binding with the same entry-point names and ``layer.MoELayer`` a
convenience wrapper that takes torch tensors. ``synth`` draws seeded synthetic
inputs. Importing this package does not load the library; the binding loads it
on first use and raises if it has not been built.
"""
__all__ = ["synth", "capi", "layer"]
