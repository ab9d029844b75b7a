"""MiTA (Mixture-of-Top-k Attention) forward pass for NVIDIA GB300 (sm_103a).

The compute path is the C-ABI library ``libmita.so`` (hand-written CUDA);
``sparse_top_landmark_gb300.mita`` is the thin Python binding over it.  The
binding is imported lazily so that ``workloads`` can be used without a GPU.
"""
import importlib

__all__ = ["mita", "workloads"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
