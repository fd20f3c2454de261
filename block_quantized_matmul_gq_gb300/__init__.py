"""block_quantized_matmul_gq_gb300 -- block-quantized (Q4_0 / Q8_0) mul_mat for GB300.

The compute path is the C-ABI library ``libgq.so`` (hand-written sm_103a kernels, declared
in ``include/gq.h``); ``binding`` is its thin Python face and loads the library on import,
raising if it has not been built -- there is no CPU fallback. ``workloads`` holds the
seeded synthetic inputs and loads nothing. Import the submodules directly:

    from block_quantized_matmul_gq_gb300 import binding, workloads
"""
