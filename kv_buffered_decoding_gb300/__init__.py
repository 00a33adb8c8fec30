"""libkvb: KV-buffered linear-attention decoding (KVBuffer) on GB300.

The compute path is the C-ABI library ``_lib/libkvb.so`` (hand-written CUDA
for sm_103a, declared in include/kvb.h); ``kvb`` is its Python binding and
``build`` compiles it.  ``inputs`` holds the seeded synthetic workloads.
Importing the package loads nothing; ``kvb.load_library()`` (called by
``kvb.Pool``) loads the library and raises if it has not been built.
"""
__version__ = "0.1.0"
