"""GB300-native (sm_103a) tensor-parallel linear block: column-parallel GEMM with
fused GELU/SwiGLU, row-parallel GEMM, and the on-device shard sum that stands in
for the all-reduce, forward and backward, with all N shards as virtual ranks on
one GPU.

The compute lives in the C-ABI library `libtpmlp.so` (CUDA kernels for sm_103a);
`attention_gemms_gb300.tpmlp` is its thin ctypes binding.
"""
__all__ = ["synth"]
