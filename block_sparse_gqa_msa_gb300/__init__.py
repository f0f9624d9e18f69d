"""GB300-native MiniMax Sparse Attention (MSA): block-sparse, causal,
document-local grouped-query attention (64 query / 4 KV / 4 index heads, head
dim 128, 128-key blocks, top-16 selection) forward and backward behind the C
ABI of libmsa.so (include/msa.h).

    from block_sparse_gqa_msa_gb300 import api
    plan = api.msa_build_plan(q2k, doc_offsets)
    o, lse = api.msa_forward(plan, q, k, v, scale)
    dq, dk, dv = api.msa_backward(plan, q, k, v, o, lse, do, scale)

Submodules: ``api`` (the binding), ``inputs`` (seeded synthetic workloads),
``build`` (in-tree nvcc build of libmsa.so).
"""
