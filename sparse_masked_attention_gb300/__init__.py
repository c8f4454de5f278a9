"""FlashMask-style exact masked attention with a column-wise sparse mask, for
GB300 (sm_103a): a C-ABI CUDA library (``include/flashmask.h``), its ctypes
binding, and a PyTorch front end.

``workloads`` (seeded inputs and mask generators) imports neither torch's CUDA
side nor the library, so it loads anywhere.
"""

__all__ = ["attention", "binding", "workloads", "build"]


def __getattr__(name):
    if name in ("fwd", "bwd", "classify", "count_unmasked", "flashmask_attention",
                "FlashMaskError", "get_error", "workspace_size"):
        from . import attention
        return getattr(attention, name)
    raise AttributeError(name)
