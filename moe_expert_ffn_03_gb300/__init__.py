"""GB300 (sm_103a) grouped MXFP8 MoE expert FFN.

The compute lives in ``libmoeffn.so`` (hand-written CUDA, C ABI declared in
``include/moe_ffn.h``).  ``binding`` wraps each C entry point under the same
name; ``layer`` allocates the buffers of one layer step with torch and calls
the entry points in order.  Importing this package does not load the library;
the first call does, and raises if it is missing.
"""
