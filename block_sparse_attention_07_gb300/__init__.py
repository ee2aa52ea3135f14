"""MiniMax Sparse Attention (MSA) decode hot path for GB300 (sm_103a).

The compute path lives in ``libmsa.so`` (hand-written CUDA behind a C ABI,
declared in include/msa.h); ``block_sparse_attention_07_gb300.msa`` is the thin
ctypes binding over it. ``synth`` draws the seeded synthetic workloads.
Importing the package loads nothing; importing ``msa`` loads the library and
fails loudly if it has not been built.
"""
