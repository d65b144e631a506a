"""GB300-native verification hot path of speculative decoding.

Two operations run as hand-written sm_103a CUDA behind a C ABI
(``include/spec_verify.h``): multi-query causal attention of the k draft
queries over a paged KV cache (``spec_verify_attn``) and greedy
longest-prefix acceptance (``spec_accept_greedy``).  The Python side is a
thin ctypes binding (:mod:`.binding`) plus the seeded input generator
(:mod:`.workload`).  Importing the package does not load the CUDA library;
the first binding call does, and fails loudly if it is missing.
"""
__version__ = "0.1.0"
