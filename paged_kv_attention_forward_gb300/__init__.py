"""GB300-native paged-KV attention: append, batched decode/verify attention, greedy accept.

The compute path is the C-ABI CUDA library ``libpkv.so`` (sm_103a kernels) behind
the ctypes binding in :mod:`paged_kv_attention_forward_gb300.pkv`.  Importing this
package loads nothing; the library is loaded on the first call and its absence is
an error (there is no CPU fallback).
"""
__all__ = ["pkv", "workloads"]
