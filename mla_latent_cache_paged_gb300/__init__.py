"""Absorbed MLA decode over a paged latent cache, for GB300 (sm_103a).

The compute lives in the C-ABI library ``libmla_decode.so`` built from
``csrc/``; ``binding`` marshals torch tensors into its calls.
"""
