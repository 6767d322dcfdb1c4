"""GB300 (sm_103a) MLA decode over an absorbed, paged latent KV cache.

The compute path is the C-ABI library ``libmla_decode.so`` built from
``csrc/``; ``binding`` wraps it with the same entry-point names.  Importing
this package does not load the library; the first call does, and raises if it
is missing.
"""
