"""invariant_selected_token_gb300 -- layout-invariant selected-token logprob on GB300.

The compute path is the C-ABI library ``librlk.so`` (hand-written sm_103a
CUDA kernels); ``invariant_selected_token_gb300.binding`` marshals torch
tensors into its calls.  Importing the package loads nothing, so the seeded
input generators (``invariant_selected_token_gb300.workloads``) work on
machines without a GPU.  Any call through the binding raises if
``librlk.so`` is missing: there is no fallback path.
"""
