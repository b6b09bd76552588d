"""Log-linear attention (Log-Linear Mamba-2 form) on GB300.

The compute path is the C-ABI library ``liblla.so`` (hand-written sm_103a
CUDA kernels); ``binding`` marshals torch tensors into its calls.
"""
