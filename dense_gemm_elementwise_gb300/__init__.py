"""GB300 (sm_103a) batched dense GEMM with a fused elementwise epilogue.

The product is the C-ABI library ``libgemm_epi.so`` (``include/gemm_epi.h``);
``binding`` is its thin ctypes front end.  ``workloads`` holds the workload
table and seeded input generators.
"""
