"""B300-native fused decode MoE layer (one persistent pass per layer).

The compute path is the CUDA library ``libmoe.so`` built from ``csrc/``; the
Python binding in ``binding`` only marshals arguments to its C ABI (declared
in ``include/moe.h``). Importing this package loads nothing; ``binding.lib()``
loads the library on first use and raises if it is missing.
"""
__all__ = ["binding", "inputs"]
