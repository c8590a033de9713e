"""GB300 (sm_103a) grouped-query attention block forward of Llama-3 / Llama-3.1 8B.

The compute lives in the C-ABI library ``libgqa_attn.so`` (include/gqa_attn.h); ``abi``
is its thin ctypes binding (argument marshalling only) and ``inputs`` draws the seeded
synthetic workloads.
"""
