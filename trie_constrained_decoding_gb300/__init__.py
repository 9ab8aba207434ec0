"""Trie-constrained greedy decoding for finite-set outputs on GB300 (sm_103a).

The compute path lives in ``libtcd.so`` (CUDA kernels + a C ABI declared in
``include/tcd.h``); ``trie_constrained_decoding_gb300.binding`` is the thin
ctypes layer over it.  ``trie_constrained_decoding_gb300.inputs`` holds the
seeded synthetic workloads.  Importing this package loads neither.
"""

__all__ = ["binding", "inputs"]
