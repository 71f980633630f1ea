"""GB300-native kvi8r K/V store and query-chunked attention.

The compute path is the C-ABI library ``libh3kv.so`` (hand-written sm_103a
CUDA kernels).  ``store_h3kv_build_gb300.binding`` is the thin Python binding
over it; importing the binding loads the library and raises if it has not been
built.  This package ``__init__`` imports nothing heavy so that the input
generator (``synth``) can be used without the library.
"""
__all__ = ["binding", "synth"]
