"""GB300-native per-block KV-cache token eviction (KNorm, Q-Filters, CurDKV-adapted).

The compute path is the C-ABI library ``libevict.so`` built from ``csrc/``;
``binding`` marshals arguments to it. Importing this package does not load
the library; ``binding.load()`` does, and raises if it is missing.
"""
__all__ = ["binding", "synth"]
