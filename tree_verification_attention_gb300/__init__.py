"""Tree-verification attention and greedy tree acceptance for GB300 (sm_103a).

The compute path is the C-ABI shared library ``libtva.so`` built from ``csrc/``;
:mod:`tree_verification_attention_gb300.api` is a thin ctypes binding over it that only
marshals torch tensors into pointers and the current CUDA stream.  Importing this
package does not load the library; the first call does, and fails loudly if the
library is missing.
"""
__all__ = ["api", "workloads"]
