"""GB300-native top-k sparse attention (DeepSeek V4 ``sparse_attn``) and the
bit-packed top-k mask builder.

The compute lives in a C-ABI shared library (``libsa.so``, built from
``csrc/`` for sm_103a); ``binding`` marshals torch tensors into it.  Import
``deepseek_top_sparse_gb300.binding`` (or the names re-exported here) to use
it; ``workloads`` only generates seeded synthetic inputs.
"""

import importlib

__all__ = ["binding", "workloads", "sparse_attn", "build_topk_mask", "topk_mask_shape"]


def __getattr__(name):
    # Lazy: importing the package (e.g. for `workloads`) must not require the
    # CUDA library; calling into it does, and fails loudly when it is missing.
    if name in ("sparse_attn", "build_topk_mask", "topk_mask_shape"):
        return getattr(importlib.import_module(__name__ + ".binding"), name)
    raise AttributeError(name)
