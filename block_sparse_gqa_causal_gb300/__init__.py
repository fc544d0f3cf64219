"""GB300-native MiniMax Sparse Attention (MSA) hot path.

The CUDA library (libmsa.so, C-ABI declared in include/msa.h) is loaded on
first use by block_sparse_gqa_causal_gb300.api; importing the package itself
loads nothing, so the input generator and workload table can be used on a
machine without a GPU.
"""
__all__ = ["api", "inputs", "workloads"]
