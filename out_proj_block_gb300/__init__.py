"""GB300-native fused decode-attention block (QKV -> KV append -> attention -> out-proj).

The compute path is the C-ABI library ``libcfa.so`` built from ``csrc/``; the
Python side (``cfa.py``) only marshals arguments. Importing this package does
not load the library: ``out_proj_block_gb300.cfa`` does, and raises if it has
not been built.
"""
__all__ = ["cfa", "workloads", "build"]
