"""GB300-native DBSCAN hot path: eps-neighbour counting over all point pairs,
core detection, union-find cluster merging and border assignment, in
hand-written sm_103a CUDA kernels behind a C ABI (``include/dbscan.h``).

The Python names mirror the C entry points; they only marshal arguments.
"""
__all__ = ["dbscan_fit", "dbscan_fit_ex", "dbscan_workspace_size", "dbscan_strerror"]


def __getattr__(name):
    if name in __all__ or name in ("DbscanError", "Status", "library_path", "load"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
