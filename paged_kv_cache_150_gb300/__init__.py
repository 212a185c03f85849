"""Paged-KV decode attention for NVIDIA GB300 (sm_103a).

The compute path is the C-ABI library ``libpa.so`` (hand-written CUDA); this
package only marshals arguments to it.  The library is loaded on first use, and
every call fails loudly when it is missing.
"""
